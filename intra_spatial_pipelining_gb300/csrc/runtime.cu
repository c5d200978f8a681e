// Host runtime of libsgp: argument validation, workspace layout, the per-op launch
// planning shared by temporal and pipelined execution, SM pools (green contexts), the
// augmented task DAG of the pipeline as an explicit CUDA graph, stage timing and the
// two-stage balancer.
//
// The execution model follows "SubGPU Pipelining: Intra-GPU Fine-Grained Spatial
// Parallelism for LLM Inference": Section 3.1 (contiguous segments bound to stages with
// disjoint SM pools, Eq. 1-3), Section 3.2 (tasks (layer, microbatch, segment) with data
// edges and per-stage FIFO edges in a fixed global dispatch order), Section 5.3 (green
// contexts for the SM pools, CUDA graphs for submission, events/graph edges for the
// producer/consumer dependencies).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_set>
#include <vector>

#include "kernels.h"
#include "sgp.h"

using namespace sgp;

// =======================================================================================
// errors
// =======================================================================================
namespace {

thread_local std::string g_err;

int fail_cuda(cudaError_t e, const char* what) {
    g_err = std::string(what) + ": " + cudaGetErrorString(e);
    return SGP_ERR_CUDA;
}
int fail_drv(CUresult r, const char* what) {
    g_err = std::string(what) + ": CUresult " + std::to_string((int)r);
    return SGP_ERR_CUDA;
}
int fail_arg(const char* what) {
    g_err = std::string("invalid argument: ") + what;
    return SGP_ERR_INVALID_ARG;
}

#define CK(x)                                          \
    do {                                               \
        cudaError_t e_ = (x);                          \
        if (e_ != cudaSuccess) return fail_cuda(e_, #x); \
    } while (0)
#define CKD(x)                                          \
    do {                                                \
        CUresult r_ = (x);                              \
        if (r_ != CUDA_SUCCESS) return fail_drv(r_, #x); \
    } while (0)

// =======================================================================================
// driver entry points (fetched at run time: the library links no libcuda)
// =======================================================================================
struct Driver {
    PFN_cuTensorMapEncodeTiled_v12000 encodeTiled = nullptr;
    PFN_cuGraphAddNode_v12030 graphAddNode = nullptr;
    PFN_cuKernelSetAttribute_v12000 kernelSetAttribute = nullptr;
    PFN_cuDeviceGetDevResource_v12040 devGetResource = nullptr;
    PFN_cuDevSmResourceSplitByCount_v12040 smSplit = nullptr;
    PFN_cuDevResourceGenerateDesc_v12040 genDesc = nullptr;
    PFN_cuGreenCtxCreate_v12040 greenCreate = nullptr;
    PFN_cuGreenCtxDestroy_v12040 greenDestroy = nullptr;
    PFN_cuCtxFromGreenCtx_v12040 ctxFromGreen = nullptr;
    PFN_cuGreenCtxGetDevResource_v12040 greenGetResource = nullptr;
    bool core = false;   // tensor maps, graph nodes, kernel attributes
    bool green = false;  // green-context API
};

template <typename F>
bool get_entry(const char* name, F& fn, unsigned ver) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, ver, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
        return false;
    fn = reinterpret_cast<F>(p);
    return true;
}

Driver& drv() {
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        d.core = get_entry("cuTensorMapEncodeTiled", d.encodeTiled, 12000) &&
                 get_entry("cuGraphAddNode", d.graphAddNode, 12030) &&
                 get_entry("cuKernelSetAttribute", d.kernelSetAttribute, 12000);
        d.green = get_entry("cuDeviceGetDevResource", d.devGetResource, 12040) &&
                  get_entry("cuDevSmResourceSplitByCount", d.smSplit, 12040) &&
                  get_entry("cuDevResourceGenerateDesc", d.genDesc, 12040) &&
                  get_entry("cuGreenCtxCreate", d.greenCreate, 12040) &&
                  get_entry("cuGreenCtxDestroy", d.greenDestroy, 12040) &&
                  get_entry("cuCtxFromGreenCtx", d.ctxFromGreen, 12040) &&
                  get_entry("cuGreenCtxGetDevResource", d.greenGetResource, 12040);
    });
    return d;
}

// Opt every kernel that asks for more than 48 KB of dynamic shared memory into the full
// 227 KB, for the runtime's launches and (through its CUkernel) for every context.
int ensure_smem_attr(const void* func, size_t smem) {
    if (smem <= 48 * 1024) return 0;
    static std::mutex mu;
    static std::unordered_set<const void*> done;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(func)) return 0;
    // the opt-in limit covers static + dynamic shared memory of a block
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return (int)e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, func);
    if (e != cudaSuccess) return (int)e;
    const int max_smem = optin - (int)fa.sharedSizeBytes;
    if ((size_t)max_smem < smem) return (int)cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return (int)e;
    Driver& d = drv();
    if (d.core) {
        cudaKernel_t k;
        if (cudaGetKernel(&k, func) == cudaSuccess)
            d.kernelSetAttribute(CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, max_smem,
                                 (CUkernel)k, (CUdevice)dev);
    }
    done.insert(func);
    return 0;
}

// =======================================================================================
// launchers
// =======================================================================================
// Every kernel of this library starts with griddepcontrol.launch_dependents and calls
// griddepcontrol.wait before it touches memory a predecessor wrote (or may still read), so
// consecutive launches may overlap their launch latency and prologue with the tail of the
// previous kernel (programmatic dependent launch).  Only launches that declare overlap_ok
// (the projection kernels and their finishing passes) use it by default: measured on the
// 36-layer slice, overlapping every kernel is slower than overlapping none.
struct StreamLauncher : Launcher {
    cudaStream_t s;
    bool pdl;
    explicit StreamLauncher(cudaStream_t st, bool programmatic = true) : s(st), pdl(programmatic) {}
    int launch(const void* func, dim3 grid, dim3 block, size_t smem, void** args,
               bool overlap_ok = false) override {
        int e = ensure_smem_attr(func, smem);
        if (e) return e;
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = (pdl && overlap_ok) ? 1 : 0;
        return (int)cudaLaunchKernelExC(&cfg, func, args);
    }
};

// Appends kernel nodes to a CUDA graph as a chain, bound to one (green) context.  When the
// only dependency of a node is the previous kernel of the same chain and `pdl` is set, the
// edge is programmatic (it fires once every CTA of that kernel has started).
struct GraphLauncher : Launcher {
    CUgraph g;
    CUcontext ctx;
    std::vector<CUgraphNode> deps;
    int pdl = 0;  // 0: off, 1: every chained kernel, 2: kernels that declare overlap_ok
    bool chained = false;  // deps holds exactly the previous kernel of this chain
    GraphLauncher(CUgraph graph, CUcontext c, int programmatic = 0)
        : g(graph), ctx(c), pdl(programmatic) {}
    int launch(const void* func, dim3 grid, dim3 block, size_t smem, void** args,
               bool overlap_ok = false) override {
        const bool prog = (pdl == 1 || (pdl == 2 && overlap_ok)) && chained && deps.size() == 1;
        CUgraphNode n;
        const int e = add(func, grid, block, smem, args, deps, prog, &n);
        if (e) return e;
        deps.assign(1, n);
        chained = true;
        return 0;
    }
    int launch_side(const void* func, dim3 grid, dim3 block, size_t smem, void** args) override {
        CUgraphNode n;
        return add(func, grid, block, smem, args, deps, false, &n);
    }
    int add(const void* func, dim3 grid, dim3 block, size_t smem, void** args,
            const std::vector<CUgraphNode>& on, bool prog, CUgraphNode* out) {
        int e = ensure_smem_attr(func, smem);
        if (e) return e;
        cudaKernel_t k;
        cudaError_t ce = cudaGetKernel(&k, func);
        if (ce != cudaSuccess) return (int)ce;
        CUgraphNodeParams np;
        memset(&np, 0, sizeof(np));
        np.type = CU_GRAPH_NODE_TYPE_KERNEL;
        np.kernel.func = nullptr;
        np.kernel.kern = (CUkernel)k;
        np.kernel.ctx = ctx;
        np.kernel.gridDimX = grid.x;
        np.kernel.gridDimY = grid.y;
        np.kernel.gridDimZ = grid.z;
        np.kernel.blockDimX = block.x;
        np.kernel.blockDimY = block.y;
        np.kernel.blockDimZ = block.z;
        np.kernel.sharedMemBytes = (unsigned)smem;
        np.kernel.kernelParams = args;
        CUgraphEdgeData ed;
        memset(&ed, 0, sizeof(ed));
        ed.from_port = CU_GRAPH_KERNEL_NODE_PORT_PROGRAMMATIC;
        ed.type = CU_GRAPH_DEPENDENCY_TYPE_PROGRAMMATIC;
        CUresult r = drv().graphAddNode(out, g, on.empty() ? nullptr : on.data(),
                                        prog ? &ed : nullptr, on.size(), &np);
        if (r != CUDA_SUCCESS) {
            g_err = "cuGraphAddNode: CUresult " + std::to_string((int)r);
            return (int)cudaErrorUnknown;
        }
        return 0;
    }
};

// =======================================================================================
// validation and launch planning
// =======================================================================================
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

constexpr int kMaxTokens = 512;  // sequences per call (attention prefix table, router groups)

int check_dims(const sgp_dims* d) {
    if (!d) return fail_arg("dims is NULL");
    if (d->head_dim != 64) return fail_arg("head_dim must be 64");
    if (d->hidden <= 0 || d->hidden % 64) return fail_arg("hidden must be a positive multiple of 64");
    if (d->inter <= 0 || d->inter % 64) return fail_arg("inter must be a positive multiple of 64");
    if (d->n_kv_heads <= 0 || d->n_q_heads <= 0 || d->n_q_heads % d->n_kv_heads)
        return fail_arg("n_q_heads must be a positive multiple of n_kv_heads");
    if (d->n_q_heads / d->n_kv_heads > 16) return fail_arg("more than 16 query heads per KV head");
    if (d->top_k < 1 || d->top_k > 8) return fail_arg("top_k must be in [1, 8]");
    if (d->n_experts < d->top_k || d->n_experts > 1024) return fail_arg("n_experts out of range");
    if (d->n_local_experts < 1 || d->n_local_experts > d->n_experts)
        return fail_arg("n_local_experts out of range");
    if (d->slot_map != 0 && d->slot_map != 1) return fail_arg("slot_map must be 0 or 1");
    if (d->path < 0 || d->path > 2) return fail_arg("path must be SGP_PATH_*");
    if (!(d->rope_theta >= 0.f)) return fail_arg("rope_theta must be >= 0");
    if (!(d->rms_eps > 0.f)) return fail_arg("rms_eps must be positive");
    if (!(d->comm_floor_us >= 0.f && d->comm_floor_us <= 1e5f) || !(d->comm_gbps >= 0.f))
        return fail_arg("comm_floor_us must be in [0, 1e5] and comm_gbps >= 0");
    // the router keeps 25 rows of H bf16 in shared memory (about 205 KB at H = 4096)
    if (d->hidden > 4096) return fail_arg("hidden above 4096 is not supported");
    return SGP_OK;
}

int cdiv(int a, int b) { return (a + b - 1) / b; }

int device_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 1;
    return n;
}

int qkv_rows(const sgp_dims& d) { return (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim; }
int q_width(const sgp_dims& d) { return d.n_q_heads * d.head_dim; }

// Fixed K split of a projection (a function of the shape only, so the fp32 summation order
// never depends on the SM pool): ~456 work units for the persistent GEMM (3 per SM of a
// 152-SM part), at least 4 k-blocks per segment.
// tiles counts (weight tile, 128-token pass) pairs of the full batch: with many tokens the
// passes alone give every SM work and no K split is needed.
// units_target: the (tile, pass, K segment) units the split aims at, about 2 per SM of the
// whole GPU (3 for the expert gate/up projection, whose many tiles balance better that way;
// measured).  Fixed numbers, so the split never depends on the pool a call runs on.
int choose_ksplit(int tiles, int kb_total, int kps, double units_target) {
    const int n_sb = cdiv(kb_total, kps);  // K segments are made of whole stage blocks
    int ks = (int)std::lround(units_target / tiles);
    ks = std::max(1, std::min(ks, n_sb / 2));
    return std::max(1, ks);
}

struct GemmShape {
    int K, rows_per_group, n_groups, m_tiles, a_tile_stride, a_second_off, ksplit;
    int kps;  // k-blocks per stage
};
// T is the full batch of the call (never the microbatch), so the K split -- and with it every
// summation order -- is the same for temporal and pipelined execution.
GemmShape gemm_shape(const sgp_dims& d, int op, int T) {
    GemmShape g{};
    switch (op) {
        case SGP_OP_QKV:
            g = {d.hidden, qkv_rows(d), 1, cdiv(qkv_rows(d), 128), 128, 64, 1};
            break;
        case SGP_OP_OPROJ:
            g = {q_width(d), d.hidden, 1, cdiv(d.hidden, 128), 128, 64, 1};
            break;
        case SGP_OP_EXPERT_UP:
            g = {d.hidden, 2 * d.inter, d.n_local_experts, d.inter / 64, 64, d.inter, 1};
            break;
        default:  // SGP_OP_EXPERT_DOWN
            g = {d.inter, d.hidden, d.n_local_experts, cdiv(d.hidden, 128), 128, 64, 1};
            break;
    }
    const bool grouped = op == SGP_OP_EXPERT_UP || op == SGP_OP_EXPERT_DOWN;
    const int rows = grouped ? cdiv(T * d.top_k, d.n_local_experts) : T;
    // a pass of 128+ tokens makes the activation rows the larger part of a stage: one k-block
    // per stage keeps the ring deep (both choices follow the full batch, like the K split)
    g.kps = rows >= 128 ? 1 : 2;
    g.ksplit = choose_ksplit(g.n_groups * g.m_tiles * cdiv(std::max(1, rows), kGemmMaxN), g.K / 64,
                             g.kps, op == SGP_OP_EXPERT_UP ? 456.0 : 304.0);
    return g;
}

bool use_tc_dense(const sgp_dims& d, int T) {
    if (d.path == SGP_PATH_GEMV) return false;
    if (d.path == SGP_PATH_TC) return true;
    return T >= std::max(1, d.gemv_max_tokens);
}
bool use_tc_expert(const sgp_dims& d, int T) {
    if (d.path == SGP_PATH_GEMV) return false;
    if (d.path == SGP_PATH_TC) return true;
    return (long)T * d.top_k >= (long)std::max(1, d.gemv_max_tokens) * d.n_local_experts;
}

int attn_smax(int max_kv) { return std::max(1, cdiv(max_kv, kAttnChunk)); }

// ---------------------------------------------------------------------------------------
// workspace layout: status | zeroed region (counters, flags) | batch-wide activations |
// per-microbatch scratch.  All offsets 256-byte aligned.
// ---------------------------------------------------------------------------------------
struct Layout {
    int T = 0, m = 1, b = 0, S_max = 1, n_flags = 0;
    size_t status = 0, zero_beg = 0, zero_end = 0;
    size_t attn_cnt = 0, router_cnt = 0, flags = 0, flag_cnt = 0, trace = 0, smmask = 0;
    int n_trace = 0;  // trace pairs (0: tracing off)
    size_t a = 0, q = 0, o = 0, h = 0, u = 0;
    size_t per_mu = 0;  // bytes of one microbatch's scratch block
    size_t mu_base = 0;
    // offsets inside a microbatch block
    size_t part_ml = 0, part_acc = 0, logits = 0, idx = 0, wts = 0, offsets = 0, pair_pos = 0,
           xperm = 0, zbuf = 0, ybuf = 0, gemm_part = 0, comm = 0;
    int max_tiles = 0;
    size_t total = 0;
};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

Layout make_layout(const sgp_dims& d, int T, int m, int max_kv, int n_flags, int n_trace = 0) {
    Layout L;
    L.T = T;
    L.m = m;
    L.b = T / m;
    L.S_max = attn_smax(max_kv);
    L.n_flags = n_flags;
    const int b = L.b, H = d.hidden, qw = q_width(d), k = d.top_k, R = b * k;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = al256(off + bytes);
        return o;
    };
    L.status = take(64);
    L.zero_beg = off;
    int max_tiles = 0;
    for (int op : {SGP_OP_QKV, SGP_OP_OPROJ, SGP_OP_EXPERT_UP, SGP_OP_EXPERT_DOWN}) {
        GemmShape g = gemm_shape(d, op, T);
        max_tiles = std::max(max_tiles, g.n_groups * g.m_tiles);
    }
    L.max_tiles = max_tiles;
    L.attn_cnt = take((size_t)m * b * d.n_kv_heads * 4);
    L.router_cnt = take((size_t)m * cdiv(b, 8) * 4);
    L.flags = take((size_t)std::max(1, n_flags) * 4);
    L.flag_cnt = take((size_t)std::max(1, n_flags) * 4);
    L.n_trace = n_trace;
    if (n_trace > 0) {
        L.trace = take((size_t)n_trace * 16);
        L.smmask = take((size_t)n_trace * 32);  // 8 x u32 per launch
    }
    L.zero_end = off;
    L.a = take((size_t)T * H * 2);
    L.q = take((size_t)T * qw * 2);
    L.o = take((size_t)T * qw * 2);
    L.h = take((size_t)T * H * 2);
    L.u = take((size_t)T * H * 2);
    // per-microbatch block
    size_t mo = 0;
    auto mtake = [&](size_t bytes) {
        size_t o = mo;
        mo = al256(mo + bytes);
        return o;
    };
    L.part_ml = mtake((size_t)b * d.n_kv_heads * L.S_max * 32 * 4);
    L.part_acc = mtake((size_t)b * d.n_kv_heads * L.S_max * 16 * 64 * 4);
    L.logits = mtake((size_t)b * d.n_experts * 4);
    L.idx = mtake((size_t)R * 4);
    L.wts = mtake((size_t)R * 4);
    L.offsets = mtake((size_t)(d.n_local_experts + 1) * 4);
    L.pair_pos = mtake((size_t)R * 4);
    L.xperm = mtake((size_t)R * H * 2);
    L.zbuf = mtake((size_t)R * d.inter * 2);
    L.ybuf = mtake((size_t)R * H * 4);
    L.comm = mtake((size_t)R * H * 2);  // virtual-communication scratch (largest payload)
    size_t gp = 0;
    for (int op : {SGP_OP_QKV, SGP_OP_OPROJ, SGP_OP_EXPERT_UP, SGP_OP_EXPERT_DOWN}) {
        GemmShape g = gemm_shape(d, op, T);
        const int rows = (op == SGP_OP_QKV || op == SGP_OP_OPROJ) ? b : R;
        gp = std::max(gp, (size_t)g.ksplit * rows * g.m_tiles * 128 * 4);
    }
    L.gemm_part = mtake(gp);
    L.per_mu = al256(mo);
    L.mu_base = off;
    L.total = L.mu_base + (size_t)m * L.per_mu;
    return L;
}

// pointers into one workspace
struct Ws {
    uint8_t* base;
    const Layout* L;
    uint32_t* status() const { return reinterpret_cast<uint32_t*>(base + L->status); }
    template <typename T>
    T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
    template <typename T>
    T* mu(int m, size_t off) const {
        return reinterpret_cast<T*>(base + L->mu_base + (size_t)m * L->per_mu + off);
    }
};

// ---------------------------------------------------------------------------------------
// tensor maps
// ---------------------------------------------------------------------------------------
// N-D bf16 tensor map with the 128-byte swizzle.  dims innermost first; strides in bytes
// for dims 1..rank-1.
int make_tmap_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides, const uint32_t* box) {
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = drv().encodeTiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
                                   const_cast<void*>(base), d, st, b, es,
                                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail_drv(r, "cuTensorMapEncodeTiled");
    return SGP_OK;
}

int make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
              uint32_t box_inner, uint32_t box_rows) {
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = drv().encodeTiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                   const_cast<void*>(base), dims, strides, box, es,
                                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail_drv(r, "cuTensorMapEncodeTiled");
    return SGP_OK;
}

// ---------------------------------------------------------------------------------------
// one op of one layer for one microbatch
// ---------------------------------------------------------------------------------------
struct RunEnv {
    const sgp_dims* d;
    const sgp_layer* layer;
    const int32_t* kv_len;
    const bf16* x_cur;  // residual input of this layer (batch-wide)
    bf16* x_out;        // residual output (batch-wide)
    int T;
    Ws ws;
    int32_t* topk_idx;  // this layer's user outputs (batch-wide) or NULL
    float* topk_w;
    bool tc_dense, tc_expert;
    int serpentine;
    int pool_sms;       // SMs of the pool the kernels run on (persistent grid size)
    // RMSNorm-1 of the next layer fused into this layer's combine (NULL: not fused), and
    // whether this layer's own RMSNorm-1 was produced by the previous layer's combine
    const sgp_layer* next = nullptr;
    bool norm_fused = false;
    // weight loads of this microbatch keep the lines in L2 for the next microbatch
    bool keep_weights = false;
    // L2 prefetch of the next projection's weights beside the chain: cap in MB for the
    // expert matrices (the dense ones are prefetched whole); < 0: off
    int prefetch_mb = -1;
    int mu = 0;
    const sgp_layer* next_layer = nullptr;  // the layer after this one (its QKV weights)
};

// The combine can produce the next layer's RMSNorm-1 while it holds the row (H <= 4096).
bool can_fuse_norm(const sgp_dims& d) { return d.hidden <= 4096; }

// After a projection's main kernel: prefetch into L2 the weights of the projection after
// it, beside the chain, so that the HBM idle time of the kernels in between (a finishing
// pass, the attention of a sliding layer, the router and dispatch, the combine) moves them.
// QKV -> output projection, output projection -> expert gate/up, expert gate/up -> expert
// down, expert down -> the next layer's QKV.  Only the timing changes.
int side_prefetch(Launcher& L, const RunEnv& e, int op, int mu, const KCtx& c) {
    if (e.prefetch_mb < 0) return 0;
    const sgp_dims& d = *e.d;
    PrefetchProblem pf;
    memset(&pf, 0, sizeof(pf));
    pf.grid = e.pool_sms;
    const size_t cap = (size_t)e.prefetch_mb << 20;
    // a serpentine microbatch walks the expert slots from the last one: take the tail
    const bool tail = e.serpentine && (mu & 1);
    auto take = [&](const void* base, size_t total, size_t limit) {
        const size_t nb = std::min(total, limit) & ~size_t(15);
        pf.base[0] = tail ? static_cast<const char*>(base) + (total - nb) : base;
        pf.bytes[0] = nb;
    };
    switch (op) {
        case SGP_OP_QKV:
            take(e.layer->w_o, (size_t)d.hidden * q_width(d) * 2, SIZE_MAX);
            pf.base[0] = e.layer->w_o;  // dense: no serpentine order
            break;
        case SGP_OP_OPROJ:
            take(e.layer->w_gate_up, (size_t)d.n_local_experts * 2 * d.inter * d.hidden * 2, cap);
            break;
        case SGP_OP_EXPERT_UP:
            take(e.layer->w_down, (size_t)d.n_local_experts * d.hidden * d.inter * 2, cap);
            break;
        default:  // SGP_OP_EXPERT_DOWN
            if (!e.next_layer) return 0;
            take(e.next_layer->w_qkv, (size_t)qkv_rows(d) * d.hidden * 2, SIZE_MAX);
            pf.base[0] = e.next_layer->w_qkv;
            break;
    }
    KCtx pc = c;
    pc.wait_flag = nullptr;
    pc.post_flag = nullptr;
    pc.post_cnt = nullptr;
    pc.trace = nullptr;
    pc.smmask = nullptr;
    pc.fault = 0;
    return enqueue_prefetch(L, pf, pc);
}

int gemm_op(Launcher& L, const RunEnv& e, int op, int mu, const KCtx& c) {
    const sgp_dims& d = *e.d;
    const int b = e.ws.L->b, row0 = mu * b, R = b * d.top_k;
    GemmShape gs = gemm_shape(d, op, e.T);
    const bool grouped = (op == SGP_OP_EXPERT_UP || op == SGP_OP_EXPERT_DOWN);
    const bool tc = grouped ? e.tc_expert : e.tc_dense;
    const bf16* W = nullptr;
    const bf16* X = nullptr;  // activation matrix base (dense: batch-wide; grouped: per mu)
    int xrows = 0;
    EpiArgs epi;
    memset(&epi, 0, sizeof(epi));
    switch (op) {
        case SGP_OP_QKV:
            W = (const bf16*)e.layer->w_qkv;
            X = e.ws.at<bf16>(e.ws.L->a);
            epi.mode = EPI_QKV;
            epi.n_out = qkv_rows(d);
            epi.q = e.ws.at<bf16>(e.ws.L->q);
            epi.q_width = q_width(d);
            epi.kc = (bf16*)e.layer->k_cache;
            epi.vc = (bf16*)e.layer->v_cache;
            epi.kv_len = e.kv_len;
            epi.nkv = d.n_kv_heads;
            epi.cap = e.layer->kv_cap;
            epi.d = d.head_dim;
            epi.rope_theta = d.rope_theta;
            if (d.rope_theta > 0.f)
                for (int i = 0; i < 32; ++i) {
                    const double f = std::pow((double)d.rope_theta, -2.0 * i / d.head_dim);
                    epi.rope_fhi[i] = (float)f;
                    epi.rope_flo[i] = (float)(f - (double)epi.rope_fhi[i]);
                }
            break;
        case SGP_OP_OPROJ:
            W = (const bf16*)e.layer->w_o;
            X = e.ws.at<bf16>(e.ws.L->o);
            epi.mode = EPI_RESID;
            epi.n_out = d.hidden;
            epi.ld = d.hidden;
            epi.resid = e.x_cur;
            epi.out = e.ws.at<bf16>(e.ws.L->h);
            break;
        case SGP_OP_EXPERT_UP:
            W = (const bf16*)e.layer->w_gate_up;
            X = e.ws.mu<bf16>(mu, e.ws.L->xperm);
            xrows = R;
            epi.mode = EPI_SWIGLU;
            epi.n_out = d.inter;
            epi.ld = d.inter;
            epi.out = e.ws.mu<bf16>(mu, e.ws.L->zbuf);
            break;
        default:
            W = (const bf16*)e.layer->w_down;
            X = e.ws.mu<bf16>(mu, e.ws.L->zbuf);
            xrows = R;
            epi.mode = EPI_F32;
            epi.n_out = d.hidden;
            epi.ld = d.hidden;
            epi.out_f32 = e.ws.mu<float>(mu, e.ws.L->ybuf);
            break;
    }
    const int* goff = grouped ? e.ws.mu<int>(mu, e.ws.L->offsets) : nullptr;
    int r0;
    if (!tc) {
        GemvProblem p;
        memset(&p, 0, sizeof(p));
        p.W = W;
        p.K = gs.K;
        p.rows_per_group = gs.rows_per_group;
        p.n_groups = gs.n_groups;
        p.n_out = (op == SGP_OP_EXPERT_UP) ? d.inter : gs.rows_per_group;
        p.swiglu = (op == SGP_OP_EXPERT_UP);
        p.up_off = d.inter;
        p.X = X;
        p.group_offsets = goff;
        p.row0 = grouped ? 0 : row0;
        p.nrows = grouped ? 0 : b;
        p.epi = epi;
        if ((r0 = enqueue_gemv(L, p, c)) != 0) return r0;
        return side_prefetch(L, e, op, mu, c);
    }
    GemmProblem p;
    memset(&p, 0, sizeof(p));
    int r;
    // tokens per accumulator pass: the whole microbatch (dense) or the expected rows of a slot
    // plus a quarter (grouped; a fuller slot takes a second pass)
    int expect = grouped ? cdiv(R, gs.n_groups) : b;
    if (grouped) expect += expect / 4;
    p.n_cap = std::min(kGemmMaxN, std::max(16, (expect + 15) & ~15));
    const uint64_t kb_total = gs.K / 64, rowb = (uint64_t)gs.K * 2;
    const uint64_t total_rows = (uint64_t)gs.n_groups * gs.rows_per_group;
    if (op == SGP_OP_EXPERT_UP) {
        // {64, row, half, k-block}: the 64 gate rows and the 64 up rows of a tile land as one
        // 128-row tile per k-block.  Rows are bounded so that row + half * I stays in range.
        const uint64_t dims[4] = {64, total_rows - (uint64_t)d.inter, 2, kb_total};
        const uint64_t str[3] = {rowb, (uint64_t)d.inter * rowb, 128};
        const uint32_t box[4] = {64, 64, 2, (uint32_t)gs.kps};
        if ((r = make_tmap_nd(&p.tmA, W, 4, dims, str, box)) != SGP_OK) return r;
        p.a_4d = 1;
    } else {
        const uint64_t dims[3] = {64, total_rows, kb_total};
        const uint64_t str[2] = {rowb, 128};
        const uint32_t box[3] = {64, 128, (uint32_t)gs.kps};
        if ((r = make_tmap_nd(&p.tmA, W, 3, dims, str, box)) != SGP_OK) return r;
        p.a_4d = 0;
    }
    {
        // activations: grouped -> the slot-sorted matrix; dense -> only this microbatch's rows
        // (the rest is out of bounds and reads as zero)
        const bf16* xb = grouped ? X : X + (size_t)row0 * gs.K;
        const uint64_t dims[3] = {64, (uint64_t)(grouped ? xrows : b), kb_total};
        const uint64_t str[2] = {rowb, 128};
        const uint32_t box[3] = {64, (uint32_t)p.n_cap, (uint32_t)gs.kps};
        if ((r = make_tmap_nd(&p.tmB, xb, 3, dims, str, box)) != SGP_OK) return r;
        // A slot that overflows a full pass by a few rows: those rows ride along with the last
        // full pass (second accumulator) instead of a pass of their own, which would stream
        // the weight tile once more.  For grouped passes capped at the MMA's 256 tokens when
        // a slot is expected to fit one pass: the tail accumulator leaves room for only one
        // accumulator buffer, so every further pass would wait for the previous one's drain
        // (measured at 512 rows per slot: expert gate/up 101 -> 125 us).  The staging chunk
        // shrinks to 32 tokens so that the ring keeps its depth.
        if (grouped && p.n_cap == kGemmMaxN && cdiv(R, gs.n_groups) <= kGemmMaxN + 16) {
            p.tail_cap = 32;
            const uint32_t box2[3] = {64, (uint32_t)p.tail_cap, (uint32_t)gs.kps};
            if ((r = make_tmap_nd(&p.tmB2, xb, 3, dims, str, box2)) != SGP_OK) return r;
        }
    }
    p.ts_rows = p.tail_cap > 0 ? 32 : kTsRows;
    p.K = gs.K;
    p.kb_total = gs.K / 64;
    p.kps = gs.kps;
    p.n_sb = cdiv(p.kb_total, p.kps);
    p.ksplit = gs.ksplit;
    p.m_tiles = gs.m_tiles;
    p.n_groups = gs.n_groups;
    p.rows_per_group = gs.rows_per_group;
    p.a_tile_stride = gs.a_tile_stride;
    p.a_second_off = gs.a_second_off;
    p.group_offsets = goff;
    p.row0 = row0;
    p.nrows = b;
    p.R = grouped ? R : b;
    const int stage_bytes = p.kps * (16384 + (p.n_cap + p.tail_cap) * 128);
    // one persistent CTA per SM: ring + accumulator staging within kGemmSmemBudget, which
    // leaves room beside it for a CTA of the small kernel before it (a programmatic launch
    // lets this kernel's CTAs start, and prefetch weights, while that kernel still runs).
    // Passes of 128+ tokens take the whole 227 KB instead: there a deep ring matters more.
    // A grouped projection follows the dispatch (a few KB) or the gate/up finishing pass
    // (none), so it keeps only that much room: one more stage at 32-token microbatches
    // (measured: 64 sequences in two microbatches, pipeline 7.88 -> 7.75 ms).
    const int budget = p.n_cap >= 128 ? 232448 : grouped ? kGemmSmemBudgetGrouped : kGemmSmemBudget;
    p.stages = std::max(2, std::min(8, (budget - 2304 - std::min(p.n_cap, p.ts_rows) * 512) /
                                          stage_bytes));
    p.ring_bytes = (int)gemm_tc_ring_bytes(p.n_cap, p.stages, p.kps, p.tail_cap, p.ts_rows);
    p.n_units = gs.n_groups * gs.m_tiles * gs.ksplit;
    p.grid = e.pool_sms;
    p.serpentine = grouped && e.serpentine && (mu & 1);
    p.keep_weights = e.keep_weights ? 1 : 0;
    p.partial = e.ws.mu<float>(mu, e.ws.L->gemm_part);
    if (p.ksplit == 1) {  // the GEMM applies the epilogue itself: one launch for the op
        p.fused_epi = 1;
        p.out_row0 = grouped ? 0 : row0;
        p.epi = epi;
        if ((r0 = enqueue_gemm_tc(L, p, c)) != 0) return r0;
        return side_prefetch(L, e, op, mu, c);
    }
    // the expert-down K segments are summed by the combine (it reads each routed row once)
    if (op == SGP_OP_EXPERT_DOWN) {
        if ((r0 = enqueue_gemm_tc(L, p, c)) != 0) return r0;
        return side_prefetch(L, e, op, mu, c);
    }
    // the flag check belongs to the first launch, the publish to the last
    KCtx c1 = c, c2 = c;
    c1.post_flag = nullptr;
    c1.post_cnt = nullptr;
    c2.wait_flag = nullptr;
    c2.fault = 0;
    if (c.trace) c2.trace = c.trace + 2;  // the finishing kernel has the op's second slot
    if (c.smmask) c2.smmask = c.smmask + 8;
    if ((r = enqueue_gemm_tc(L, p, c1)) != 0) return r;
    if ((r = side_prefetch(L, e, op, mu, c1)) != 0) return r;
    FinishProblem f;
    memset(&f, 0, sizeof(f));
    f.partial = p.partial;
    f.ksplit = p.ksplit;
    f.m_tiles = p.m_tiles;
    f.R = p.R;
    f.rows = p.R;
    f.out_row0 = grouped ? 0 : row0;
    f.epi = epi;
    return enqueue_gemm_finish(L, f, c2);
}

// Virtual communication (sgp_dims::comm_floor_us / comm_gbps): on when both are positive.
bool comm_on(const sgp_dims& d) { return d.comm_floor_us > 0.f && d.comm_gbps > 0.f; }
unsigned long long comm_floor_ns(const sgp_dims& d, size_t bytes) {
    return (unsigned long long)((double)d.comm_floor_us * 1e3 + (double)bytes / (double)d.comm_gbps);
}
// An op followed (or preceded) by a communication kernel: the op's first launch checks the
// handoff flag and the last one publishes it; the communication kernel has no trace slot.
void split_for_comm(const KCtx& c, bool comm_last, KCtx& op_ctx, KCtx& comm_ctx) {
    op_ctx = c;
    comm_ctx = c;
    comm_ctx.trace = nullptr;
    comm_ctx.smmask = nullptr;
    if (comm_last) {
        op_ctx.post_flag = nullptr;
        op_ctx.post_cnt = nullptr;
        op_ctx.fault &= ~FAULT_SKIP_PUBLISH;
        comm_ctx.wait_flag = nullptr;
        comm_ctx.fault &= FAULT_SKIP_PUBLISH;
    } else {
        comm_ctx.post_flag = nullptr;
        comm_ctx.post_cnt = nullptr;
        comm_ctx.fault = 0;
        op_ctx.wait_flag = nullptr;
    }
}

int enqueue_op(Launcher& L, const RunEnv& e, int op, int mu, const KCtx& c) {
    const sgp_dims& d = *e.d;
    const Layout& Lay = *e.ws.L;
    const int b = Lay.b, row0 = mu * b;
    int r = 0;
    switch (op) {
        case SGP_OP_RMSNORM_ATTN: {
            if (e.norm_fused) return 0;  // written by the previous layer's combine
            NormProblem p{e.x_cur, (const bf16*)e.layer->g_attn, e.ws.at<bf16>(Lay.a), row0, b,
                          d.hidden, d.rms_eps};
            return enqueue_rmsnorm(L, p, c);
        }
        case SGP_OP_OPROJ:
            if (comm_on(d)) {
                // attention all-reduce of the projected rows (b x H bf16)
                KCtx co, cc;
                split_for_comm(c, true, co, cc);
                if ((r = gemm_op(L, e, op, mu, co)) != 0) return r;
                const size_t bytes = (size_t)b * d.hidden * 2;
                CommProblem cp{e.ws.at<bf16>(Lay.h) + (size_t)row0 * d.hidden,
                               e.ws.mu<bf16>(mu, Lay.comm), bytes, comm_floor_ns(d, bytes)};
                return enqueue_comm(L, cp, cc);
            }
            return gemm_op(L, e, op, mu, c);
        case SGP_OP_QKV:
        case SGP_OP_EXPERT_UP:
        case SGP_OP_EXPERT_DOWN:
            return gemm_op(L, e, op, mu, c);
        case SGP_OP_ATTENTION: {
            AttnProblem p;
            memset(&p, 0, sizeof(p));
            const uint64_t rows = (uint64_t)e.T * d.n_kv_heads * e.layer->kv_cap;
            {
                const int span0 = e.layer->window > 0 ? std::min(e.layer->window, e.layer->kv_cap)
                                                      : e.layer->kv_cap;
                p.pos = attn_stage_pos((long long)e.T * d.n_kv_heads * cdiv(span0, kAttnChunk));
            }
            if ((r = make_tmap(&p.tmK, e.layer->k_cache, 64, rows, 64, p.pos)) != SGP_OK) return r;
            if ((r = make_tmap(&p.tmV, e.layer->v_cache, 64, rows, 64, p.pos)) != SGP_OK) return r;
            p.q = e.ws.at<bf16>(Lay.q);
            p.kv_len = e.kv_len;
            p.o = e.ws.at<bf16>(Lay.o);
            p.part_ml = e.ws.mu<float>(mu, Lay.part_ml);
            p.part_acc = e.ws.mu<float>(mu, Lay.part_acc);
            p.cnt = e.ws.at<uint32_t>(Lay.attn_cnt) + (size_t)mu * b * d.n_kv_heads;
            p.row0 = row0;
            p.nrows = b;
            p.nq = d.n_q_heads;
            p.nkv = d.n_kv_heads;
            p.G = d.n_q_heads / d.n_kv_heads;
            p.cap = e.layer->kv_cap;
            p.window = e.layer->window;
            p.chunk = kAttnChunk;
            const int span = e.layer->window > 0 ? std::min(e.layer->window, e.layer->kv_cap)
                                                 : e.layer->kv_cap;
            p.S_max = attn_smax(span);
            if (p.S_max > Lay.S_max) return fail_arg("kv_cap exceeds the workspace's max_kv_len");
            p.scale_log2 = 1.4426950408889634f / sqrtf((float)d.head_dim);
            p.n_cta = e.pool_sms;
            // split refills: alone on the GPU, or with 128-position stages; with 64-position
            // stages on a partial pool the joint schedule leaves more HBM to the other stage
            p.kv_split = (p.pos == 128 || e.pool_sms >= device_sms()) ? 1 : 0;
            return enqueue_attention(L, p, c);
        }
        case SGP_OP_ROUTER: {
            RouterProblem p;
            memset(&p, 0, sizeof(p));
            p.h = e.ws.at<bf16>(Lay.h);
            p.g = (const bf16*)e.layer->g_mlp;
            p.u = e.ws.at<bf16>(Lay.u);
            p.Wr = (const bf16*)e.layer->w_router;
            p.bias = e.layer->router_bias;
            p.logits = e.ws.mu<float>(mu, Lay.logits);
            p.idx = e.ws.mu<int>(mu, Lay.idx);
            p.wts = e.ws.mu<float>(mu, Lay.wts);
            p.user_idx = e.topk_idx;
            p.user_w = e.topk_w;
            p.cnt = e.ws.at<uint32_t>(Lay.router_cnt) + (size_t)mu * cdiv(b, 8);
            p.row0 = row0;
            p.nrows = b;
            p.H = d.hidden;
            p.E = d.n_experts;
            p.k = d.top_k;
            p.eps = d.rms_eps;
            return enqueue_router(L, p, c);
        }
        case SGP_OP_DISPATCH: {
            DispatchProblem p{e.ws.mu<int>(mu, Lay.idx), e.ws.at<bf16>(Lay.u),
                              e.ws.mu<bf16>(mu, Lay.xperm), e.ws.mu<int>(mu, Lay.offsets),
                              e.ws.mu<int>(mu, Lay.pair_pos), row0, b, d.top_k, d.hidden,
                              d.n_experts, d.n_local_experts, d.slot_map};
            if (comm_on(d)) {
                // MoE dispatch: the routed rows (b k x H bf16)
                KCtx co, cc;
                split_for_comm(c, true, co, cc);
                if ((r = enqueue_dispatch(L, p, co)) != 0) return r;
                const size_t bytes = (size_t)b * d.top_k * d.hidden * 2;
                CommProblem cp{e.ws.mu<bf16>(mu, Lay.xperm), e.ws.mu<bf16>(mu, Lay.comm), bytes,
                               comm_floor_ns(d, bytes)};
                return enqueue_comm(L, cp, cc);
            }
            return enqueue_dispatch(L, p, c);
        }
        case SGP_OP_COMBINE: {
            // a K-split tensor-core expert-down projection leaves its segments in the partial
            // buffer (no finishing pass); otherwise its rows are in ybuf
            const int ks = e.tc_expert ? gemm_shape(d, SGP_OP_EXPERT_DOWN, e.T).ksplit : 1;
            CombineProblem p{e.ws.at<bf16>(Lay.h),
                             ks > 1 ? e.ws.mu<float>(mu, Lay.gemm_part) : e.ws.mu<float>(mu, Lay.ybuf),
                             ks, b * d.top_k,
                             e.ws.mu<float>(mu, Lay.wts), e.ws.mu<int>(mu, Lay.pair_pos),
                             e.x_out, row0, b, d.top_k, d.hidden,
                             e.next ? (const bf16*)e.next->g_attn : nullptr,
                             e.next ? e.ws.at<bf16>(Lay.a) : nullptr, d.rms_eps};
            if (comm_on(d)) {
                // MoE combine: the expert outputs return (b k x H, bf16-sized payload)
                KCtx co, cc;
                split_for_comm(c, false, co, cc);
                const size_t bytes = (size_t)b * d.top_k * d.hidden * 2;
                CommProblem cp{p.Y, e.ws.mu<bf16>(mu, Lay.comm), bytes, comm_floor_ns(d, bytes)};
                if ((r = enqueue_comm(L, cp, cc)) != 0) return r;
                return enqueue_combine(L, p, co);
            }
            return enqueue_combine(L, p, c);
        }
        default:
            return fail_arg("op index");
    }
}

int check_layer(const sgp_dims& d, const sgp_layer* l, int T) {
    if (!l) return fail_arg("layer is NULL");
    const void* ptrs[] = {l->g_attn, l->w_qkv, l->w_o, l->g_mlp, l->w_router,
                          l->w_gate_up, l->w_down, l->k_cache, l->v_cache};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return fail_arg("layer pointer NULL or not 16-byte aligned");
    if (l->kv_cap < 1) return fail_arg("kv_cap must be positive");
    if (l->window < 0) return fail_arg("window must be >= 0");
    if ((uint64_t)T * d.n_kv_heads * l->kv_cap >= (1ull << 31))
        return fail_arg("KV cache rows exceed 2^31");
    return SGP_OK;
}

int status_to_code(uint32_t s) {
    if (s & ST_TIMEOUT) return SGP_ERR_TIMEOUT;
    if (s & ST_HANDOFF) return SGP_ERR_HANDOFF;
    if (s & ST_BOUNDS) return SGP_ERR_DEVICE_BOUNDS;
    return SGP_OK;
}

KCtx plain_ctx(uint32_t* status, uint64_t timeout, uint32_t tag) {
    KCtx c;
    memset(&c, 0, sizeof(c));
    c.status = status;
    c.timeout_ns = timeout;
    c.tag = tag;
    return c;
}

constexpr uint64_t kDefaultTimeout = 2000000000ull;

int run_layer_stream(const sgp_dims& d, const sgp_layer* layer, int li, const int32_t* kv_len,
                     const bf16* x_cur, bf16* x_out, int T, int32_t* tki, float* tkw, Ws ws,
                     cudaStream_t s, const sgp_layer* next, bool norm_fused) {
    StreamLauncher L(s);
    RunEnv e{&d, layer, kv_len, x_cur, x_out, T, ws, tki, tkw, use_tc_dense(d, T),
             use_tc_expert(d, T), 0, device_sms()};
    e.next = next;
    e.norm_fused = norm_fused;
    for (int op = 0; op < SGP_N_OPS; ++op) {
        KCtx c = plain_ctx(ws.status(), kDefaultTimeout, ((uint32_t)op << 24) | ((uint32_t)li << 12));
        int r = enqueue_op(L, e, op, 0, c);
        if (r == SGP_ERR_INVALID_ARG || r == SGP_ERR_CUDA) return r;
        if (r != 0) return fail_cuda((cudaError_t)r, "kernel launch");
    }
    return SGP_OK;
}

}  // namespace

// =======================================================================================
// C ABI: info
// =======================================================================================
extern "C" const char* sgp_status_string(int s) {
    switch (s) {
        case SGP_OK: return "ok";
        case SGP_ERR_INVALID_ARG: return "invalid argument";
        case SGP_ERR_UNSUPPORTED: return "unsupported device or feature";
        case SGP_ERR_CUDA: return "CUDA error";
        case SGP_ERR_TIMEOUT: return "device wait timed out";
        case SGP_ERR_OOM: return "out of memory";
        case SGP_ERR_HANDOFF: return "stage handoff check failed";
        case SGP_ERR_DEVICE_BOUNDS: return "device index out of range (skipped)";
        default: return "unknown status";
    }
}

extern "C" const char* sgp_last_error(void) { return g_err.c_str(); }

extern "C" int sgp_device_info_get(sgp_device_info* info) {
    if (!info) return fail_arg("info is NULL");
    memset(info, 0, sizeof(*info));
    int dev = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&info->sm_count, cudaDevAttrMultiProcessorCount, dev));
    CK(cudaDeviceGetAttribute(&info->cc_major, cudaDevAttrComputeCapabilityMajor, dev));
    CK(cudaDeviceGetAttribute(&info->cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
    int l2 = 0;
    CK(cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev));
    info->l2_bytes = (size_t)l2;
    Driver& d = drv();
    if (d.green) {
        CK(cudaFree(0));
        CUdevResource res;
        memset(&res, 0, sizeof(res));
        if (d.devGetResource((CUdevice)dev, &res, CU_DEV_RESOURCE_TYPE_SM) == CUDA_SUCCESS) {
            info->green_ctx_supported = 1;
            info->sm_min_partition = (int)res.sm.minSmPartitionSize;
            info->sm_alignment = (int)res.sm.smCoscheduledAlignment;
        }
    }
    return SGP_OK;
}

// =======================================================================================
// C ABI: temporal execution
// =======================================================================================
extern "C" size_t sgp_workspace_bytes(const sgp_dims* d, int n_tokens, int max_kv_len) {
    if (check_dims(d) != SGP_OK || n_tokens < 1 || max_kv_len < 1) return 0;
    return make_layout(*d, n_tokens, 1, max_kv_len, 0).total;
}

static int temporal_common(const sgp_dims* d, const sgp_layer* layers, int n_layers,
                           const int32_t* kv_len, const void* x_in, void* x_out, int T,
                           int32_t* tki, float* tkw, void* ws, size_t ws_bytes,
                           const sgp_layer_dump* dump, cudaStream_t s) {
    int r;
    if ((r = check_dims(d)) != SGP_OK) return r;
    if (T < 1 || T > kMaxTokens) return fail_arg("n_tokens must be in [1, 512]");
    if (d->rope_theta > 0.f && !use_tc_dense(*d, T))
        return fail_arg("RoPE needs the tensor-core QKV path");
    if (n_layers < 1 || !layers) return fail_arg("no layers");
    if (!kv_len || !x_in || !x_out || !ws) return fail_arg("NULL pointer");
    if (!aligned16(x_in) || !aligned16(x_out) || (reinterpret_cast<uintptr_t>(ws) & 255))
        return fail_arg("x must be 16-byte and workspace 256-byte aligned");
    int max_cap = 1;
    for (int l = 0; l < n_layers; ++l) {
        if ((r = check_layer(*d, &layers[l], T)) != SGP_OK) return r;
        max_cap = std::max(max_cap, layers[l].kv_cap);
    }
    Layout Lay = make_layout(*d, T, 1, max_cap, 0);
    if (ws_bytes < Lay.total) return fail_arg("workspace too small");
    if (!drv().core) {
        g_err = "CUDA driver entry points unavailable";
        return SGP_ERR_UNSUPPORTED;
    }
    Ws w{(uint8_t*)ws, &Lay};
    CK(cudaMemsetAsync(w.base + Lay.zero_beg, 0, Lay.zero_end - Lay.zero_beg, s));
    for (int l = 0; l < n_layers; ++l) {
        const bf16* xc = (const bf16*)(l == 0 ? x_in : x_out);
        int32_t* ti = tki ? tki + (size_t)l * T * d->top_k : nullptr;
        float* tw = tkw ? tkw + (size_t)l * T * d->top_k : nullptr;
        const bool fuse = can_fuse_norm(*d);
        const sgp_layer* next = (fuse && l + 1 < n_layers) ? &layers[l + 1] : nullptr;
        if ((r = run_layer_stream(*d, &layers[l], l, kv_len, xc, (bf16*)x_out, T, ti, tw, w, s,
                                  next, fuse && l > 0)) != SGP_OK)
            return r;
    }
    if (dump) {
        const size_t H = d->hidden, qw = q_width(*d), R = (size_t)T * d->top_k;
        auto cp = [&](void* dst, const void* src, size_t bytes) -> int {
            if (dst) CK(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s));
            return SGP_OK;
        };
        if ((r = cp(dump->a, w.base + Lay.a, T * H * 2))) return r;
        if ((r = cp(dump->q, w.base + Lay.q, T * qw * 2))) return r;
        if ((r = cp(dump->o, w.base + Lay.o, T * qw * 2))) return r;
        if ((r = cp(dump->h, w.base + Lay.h, T * H * 2))) return r;
        if ((r = cp(dump->u, w.base + Lay.u, T * H * 2))) return r;
        if ((r = cp(dump->logits, w.mu<float>(0, Lay.logits), (size_t)T * d->n_experts * 4))) return r;
        if ((r = cp(dump->slot_offsets, w.mu<int>(0, Lay.offsets), (d->n_local_experts + 1) * 4)))
            return r;
        if ((r = cp(dump->pair_pos, w.mu<int>(0, Lay.pair_pos), R * 4))) return r;
        if ((r = cp(dump->z, w.mu<bf16>(0, Lay.zbuf), R * d->inter * 2))) return r;
        const GemmShape gd = gemm_shape(*d, SGP_OP_EXPERT_DOWN, T);
        if (dump->y && use_tc_expert(*d, T) && gd.ksplit > 1) {
            // the combine summed the expert-down K segments itself; form y for the dump
            FinishProblem f;
            memset(&f, 0, sizeof(f));
            f.partial = w.mu<float>(0, Lay.gemm_part);
            f.ksplit = gd.ksplit;
            f.m_tiles = gd.m_tiles;
            f.R = (int)R;
            f.rows = (int)R;
            f.epi.mode = EPI_F32;
            f.epi.n_out = (int)H;
            f.epi.ld = (int)H;
            f.epi.out_f32 = (float*)dump->y;
            StreamLauncher L(s);
            KCtx c = plain_ctx(w.status(), kDefaultTimeout, (uint32_t)SGP_OP_EXPERT_DOWN << 24);
            const int e2 = enqueue_gemm_finish(L, f, c);
            if (e2 != 0) return fail_cuda((cudaError_t)e2, "dump of y");
        } else if ((r = cp(dump->y, w.mu<float>(0, Lay.ybuf), R * H * 4))) {
            return r;
        }
    }
    return SGP_OK;
}

extern "C" int sgp_layer_temporal(const sgp_dims* d, const sgp_layer* layer, const int32_t* kv_len,
                                  const void* x_in, void* x_out, int n_tokens, int32_t* topk_idx,
                                  float* topk_w, void* ws, size_t ws_bytes,
                                  const sgp_layer_dump* dump, sgp_stream_t stream) {
    return temporal_common(d, layer, 1, kv_len, x_in, x_out, n_tokens, topk_idx, topk_w, ws,
                           ws_bytes, dump, (cudaStream_t)stream);
}

extern "C" int sgp_stack_temporal(const sgp_dims* d, const sgp_layer* layers, int n_layers,
                                  const int32_t* kv_len, const void* x_in, void* x_out,
                                  int n_tokens, int32_t* topk_idx, float* topk_w, void* ws,
                                  size_t ws_bytes, sgp_stream_t stream) {
    return temporal_common(d, layers, n_layers, kv_len, x_in, x_out, n_tokens, topk_idx, topk_w,
                           ws, ws_bytes, nullptr, (cudaStream_t)stream);
}

extern "C" int sgp_layer_op(const sgp_dims* d, const sgp_layer* layer, int op,
                            const int32_t* kv_len, const void* x_in, void* x_out, int n_tokens,
                            void* ws, size_t ws_bytes, sgp_stream_t stream) {
    int r;
    if ((r = check_dims(d)) != SGP_OK) return r;
    if (op < 0 || op >= SGP_N_OPS) return fail_arg("op index");
    if (n_tokens < 1 || n_tokens > kMaxTokens) return fail_arg("n_tokens must be in [1, 512]");
    if (d->rope_theta > 0.f && !use_tc_dense(*d, n_tokens))
        return fail_arg("RoPE needs the tensor-core QKV path");
    if (!kv_len || !x_in || !x_out || !ws) return fail_arg("NULL pointer");
    if ((reinterpret_cast<uintptr_t>(ws) & 255) || !aligned16(x_in) || !aligned16(x_out))
        return fail_arg("alignment");
    if ((r = check_layer(*d, layer, n_tokens)) != SGP_OK) return r;
    Layout Lay = make_layout(*d, n_tokens, 1, layer->kv_cap, 0);
    if (ws_bytes < Lay.total) return fail_arg("workspace too small");
    if (!drv().core) return SGP_ERR_UNSUPPORTED;
    Ws w{(uint8_t*)ws, &Lay};
    StreamLauncher L((cudaStream_t)stream);
    RunEnv e{d, layer, kv_len, (const bf16*)x_in, (bf16*)x_out, n_tokens, w, nullptr, nullptr,
             use_tc_dense(*d, n_tokens), use_tc_expert(*d, n_tokens), 0, device_sms()};
    KCtx c = plain_ctx(w.status(), kDefaultTimeout, (uint32_t)op << 24);
    r = enqueue_op(L, e, op, 0, c);
    if (r == SGP_ERR_INVALID_ARG || r == SGP_ERR_CUDA) return r;
    if (r != 0) return fail_cuda((cudaError_t)r, "kernel launch");
    return SGP_OK;
}

extern "C" int sgp_status_from_workspace(const void* ws, sgp_stream_t stream) {
    if (!ws) return fail_arg("workspace is NULL");
    uint32_t st[4] = {0, 0, 0, 0};
    CK(cudaStreamSynchronize((cudaStream_t)stream));
    CK(cudaMemcpy(st, ws, sizeof(st), cudaMemcpyDeviceToHost));
    CK(cudaMemset(const_cast<void*>(ws), 0, sizeof(st)));
    if (st[0]) {
        char buf[96];
        snprintf(buf, sizeof(buf), "device status 0x%x at op %u layer %u micro %u (detail %u)",
                 st[0], st[1] >> 24, (st[1] >> 12) & 0xFFF, st[1] & 0xFFF, st[2]);
        g_err = buf;
    }
    return status_to_code(st[0]);
}

// =======================================================================================
// C ABI: pipeline
// =======================================================================================
struct PTask {
    int stage, mu;
    int l0, op0, l1, op1;      // first and last (layer, op), inclusive, along the chain
    int pred_data, pred_stage;
};

struct sgp_pipeline {
    sgp_dims dims;
    int n_stages = 1, micro = 1, max_tokens = 0, max_kv = 0;
    sgp_pipeline_opts opts;
    int stage_of_op[2][SGP_N_OPS];
    int split[3] = {0, 0, 0};
    int dev = 0;
    CUgreenCtx gctx[4] = {nullptr, nullptr, nullptr, nullptr};
    CUcontext sctx[3] = {nullptr, nullptr, nullptr};
    int n_gctx = 0;
    uint8_t* ws = nullptr;
    size_t ws_bytes = 0;
    int ws_T = 0, ws_nflags = 0;
    Layout lay;
    // graph cache
    cudaGraphExec_t exec = nullptr;
    std::vector<uint8_t> key;
    std::vector<PTask> tasks;
    cudaStream_t last_stream = nullptr;
    int trace_pairs = 0;  // launch-trace pairs the cached graph writes
    // completion of the last run (recorded on its stream after its status copy) and a pinned
    // host copy of the device status word as that run left it
    cudaEvent_t done = nullptr;
    uint32_t* host_status = nullptr;
    bool launched = false;
};

namespace {

std::vector<PTask> build_tasks(const sgp_pipeline& p, const sgp_layer* layers, int n_layers, int m) {
    std::vector<PTask> per;
    std::vector<std::vector<int>> chain(m);
    // tasks of each microbatch along its chain
    std::vector<PTask> all;
    std::vector<long> first_pos;
    for (int mu = 0; mu < m; ++mu) {
        int cur = -1;
        for (int l = 0; l < n_layers; ++l) {
            const int sl = layers[l].window > 0 ? 1 : 0;
            for (int op = 0; op < SGP_N_OPS; ++op) {
                const int st = p.stage_of_op[sl][op];
                if (cur >= 0 && all[cur].stage == st) {
                    all[cur].l1 = l;
                    all[cur].op1 = op;
                } else {
                    PTask t{st, mu, l, op, l, op, cur, -1};
                    all.push_back(t);
                    first_pos.push_back((long)l * SGP_N_OPS + op);
                    cur = (int)all.size() - 1;
                }
            }
        }
    }
    // global dispatch order: by chain position of the first op, then microbatch
    std::vector<int> order(all.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        if (first_pos[a] != first_pos[b]) return first_pos[a] < first_pos[b];
        return all[a].mu < all[b].mu;
    });
    std::vector<int> newidx(all.size());
    for (size_t i = 0; i < order.size(); ++i) newidx[order[i]] = (int)i;
    std::vector<PTask> out(all.size());
    // one FIFO per stage, or (stage_lanes = 2) one per stage and microbatch parity: the
    // stage's two lanes share its SM pool, as two streams of one green context do
    const int lanes = p.opts.stage_lanes == 2 ? 2 : 1;
    int last_on_lane[4][2] = {{-1, -1}, {-1, -1}, {-1, -1}, {-1, -1}};
    for (size_t i = 0; i < order.size(); ++i) {
        PTask t = all[order[i]];
        t.pred_data = t.pred_data >= 0 ? newidx[t.pred_data] : -1;
        int& last = last_on_lane[t.stage][t.mu % lanes];
        t.pred_stage = last;
        last = (int)i;
        out[i] = t;
    }
    return out;
}

int ensure_ws(sgp_pipeline* p, int T, int nflags, int ntrace = 0) {
    if (p->ws && p->ws_T == T && p->ws_nflags >= nflags && p->lay.n_trace >= ntrace)
        return SGP_OK;
    if (p->ws) {
        cudaFree(p->ws);
        p->ws = nullptr;
    }
    Layout L = make_layout(p->dims, T, T / p->micro, p->max_kv, nflags, ntrace);
    cudaError_t e = cudaMalloc(&p->ws, L.total);
    if (e != cudaSuccess) {
        g_err = std::string("cudaMalloc: ") + cudaGetErrorString(e);
        return SGP_ERR_OOM;
    }
    e = cudaMemset(p->ws, 0, L.total);
    if (e != cudaSuccess) {
        cudaFree(p->ws);
        p->ws = nullptr;
        return fail_cuda(e, "cudaMemset");
    }
    p->lay = L;
    p->ws_bytes = L.total;
    p->ws_T = T;
    p->ws_nflags = nflags;
    return SGP_OK;
}

// Builds the graph of the given tasks.  stage_only >= 0 keeps only that stage's tasks and
// drops their cross-stage data edges (used for timing one stage alone).
// zero_first: the graph starts with a memset node that clears the workspace's zeroed region
// (counters, flags, trace); without it the caller clears that region before launching.
int build_graph(sgp_pipeline* p, const std::vector<PTask>& tasks, const sgp_layer* layers,
                const int32_t* kv_len, const void* x_in, void* x_out, int T, int32_t* tki,
                float* tkw, int stage_only, cudaGraph_t* out_graph, bool zero_first = true) {
    const sgp_dims& d = p->dims;
    cudaGraph_t g;
    CK(cudaGraphCreate(&g, 0));
    Ws w{p->ws, &p->lay};
    cudaGraphNode_t zero;
    cudaMemsetParams ms;
    memset(&ms, 0, sizeof(ms));
    ms.dst = p->ws + p->lay.zero_beg;
    ms.value = 0;
    ms.elementSize = 1;
    ms.width = p->lay.zero_end - p->lay.zero_beg;
    ms.height = 1;
    ms.pitch = 0;
    cudaError_t ce = zero_first ? cudaGraphAddMemsetNode(&zero, g, nullptr, 0, &ms) : cudaSuccess;
    if (ce != cudaSuccess) {
        cudaGraphDestroy(g);
        return fail_cuda(ce, "cudaGraphAddMemsetNode");
    }
    std::vector<CUgraphNode> last(tasks.size(), nullptr);
    const bool tcd = use_tc_dense(d, T), tce = use_tc_expert(d, T);
    // Layer l's RMSNorm-1 comes from layer l-1's combine unless it is the last op of its task
    // (the task's last kernel publishes the stage handoff flag, so it must be launched).
    int n_layers = 0;
    for (const PTask& t : tasks) n_layers = std::max(n_layers, t.l1 + 1);
    std::vector<char> fused(n_layers + 1, 0);
    if (can_fuse_norm(d))
        for (int l = 1; l < n_layers; ++l) {
            fused[l] = 1;
            for (const PTask& t : tasks)
                if (t.mu == 0 && t.l1 == l && t.op1 == 0) fused[l] = 0;
        }
    const uint64_t timeout = p->opts.wait_timeout_ns ? p->opts.wait_timeout_ns : kDefaultTimeout;
    uint32_t* flags = w.at<uint32_t>(p->lay.flags);
    uint32_t* fcnt = w.at<uint32_t>(p->lay.flag_cnt);
    for (size_t i = 0; i < tasks.size(); ++i) {
        const PTask& t = tasks[i];
        if (stage_only >= 0 && t.stage != stage_only) continue;
        GraphLauncher L((CUgraph)g, p->sctx[t.stage],
                        p->opts.programmatic_launch < 0 ? 0 : (p->opts.programmatic_launch == 1 ? 1 : 2));
        const bool keep_data = stage_only < 0;
        if (keep_data && t.pred_data >= 0) L.deps.push_back(last[t.pred_data]);
        if (t.pred_stage >= 0 && last[t.pred_stage]) L.deps.push_back(last[t.pred_stage]);
        if (L.deps.empty() && zero_first) L.deps.push_back((CUgraphNode)zero);
        int l = t.l0, op = t.op0;
        bool first = true;
        while (true) {
            const bool lastop = (l == t.l1 && op == t.op1);
            KCtx c = plain_ctx(w.status(), timeout,
                               ((uint32_t)op << 24) | ((uint32_t)l << 12) | (uint32_t)t.mu);
            if (first && keep_data && t.pred_data >= 0) c.wait_flag = flags + t.pred_data;
            if (lastop) {
                c.post_flag = flags + i;
                c.post_cnt = fcnt + i;
                if ((p->opts.fault_inject & 1u) && (int)i == p->opts.fault_task)
                    c.fault |= FAULT_SKIP_PUBLISH;
            }
            if ((p->opts.fault_inject & 2u) && i == 0 && op == SGP_OP_QKV) c.fault |= FAULT_DROP_TMA;
            if (p->lay.n_trace > 0) {
                const size_t ent = ((size_t)l * p->lay.m + t.mu) * SGP_N_OPS + op;
                c.trace = w.at<unsigned long long>(p->lay.trace) + 4 * ent;
                c.smmask = w.at<uint32_t>(p->lay.smmask) + 16 * ent;
            }
            RunEnv e{&d, &layers[l], kv_len, (const bf16*)(l == 0 ? x_in : x_out), (bf16*)x_out, T,
                     w, tki ? tki + (size_t)l * T * d.top_k : nullptr,
                     tkw ? tkw + (size_t)l * T * d.top_k : nullptr, tcd, tce,
                     p->opts.serpentine_experts,
                     p->sctx[t.stage] ? p->split[t.stage] : device_sms()};
            e.next = fused[l + 1] ? &layers[l + 1] : nullptr;
            e.norm_fused = fused[l] != 0;
            e.keep_weights = p->opts.weight_reuse > 0 && t.mu + 1 < p->lay.m;
            e.prefetch_mb = p->opts.l2_prefetch_mb > 0 ? p->opts.l2_prefetch_mb : -1;
            e.mu = t.mu;
            e.next_layer = l + 1 < n_layers ? &layers[l + 1] : nullptr;
            if (op == SGP_OP_RMSNORM_ATTN && e.norm_fused) {  // nothing to launch
                if (++op == SGP_N_OPS) {
                    op = 0;
                    ++l;
                }
                continue;
            }
            int r = enqueue_op(L, e, op, t.mu, c);
            if (r != 0) {
                cudaGraphDestroy(g);
                if (r == SGP_ERR_INVALID_ARG || r == SGP_ERR_CUDA) return r;
                return fail_cuda((cudaError_t)r, "graph kernel node");
            }
            first = false;
            if (lastop) break;
            if (++op == SGP_N_OPS) {
                op = 0;
                ++l;
            }
        }
        last[i] = L.deps[0];
    }
    *out_graph = g;
    return SGP_OK;
}

int setup_green(sgp_pipeline* p) {
    Driver& d = drv();
    if (!d.green) {
        g_err = "green-context driver API unavailable";
        return SGP_ERR_UNSUPPORTED;
    }
    CK(cudaFree(0));
    CUdevResource cur;
    memset(&cur, 0, sizeof(cur));
    CKD(d.devGetResource((CUdevice)p->dev, &cur, CU_DEV_RESOURCE_TYPE_SM));
    for (int s = 0; s < p->n_stages; ++s) {
        const bool lastst = (s == p->n_stages - 1);
        CUdevResource grp, rest;
        memset(&grp, 0, sizeof(grp));
        memset(&rest, 0, sizeof(rest));
        if (lastst && (int)cur.sm.smCount == p->split[s]) {
            grp = cur;
        } else {
            unsigned nb = 1;
            CKD(d.smSplit(&grp, &nb, &cur, &rest, (unsigned)p->opts.green_ctx_flags,
                          (unsigned)p->split[s]));
            if (nb != 1 || (int)grp.sm.smCount != p->split[s]) {
                g_err = "SM split of " + std::to_string(p->split[s]) + " gave " +
                        std::to_string(grp.sm.smCount) + " SMs";
                return SGP_ERR_INVALID_ARG;
            }
        }
        CUdevResourceDesc desc;
        CKD(d.genDesc(&desc, &grp, 1));
        CKD(d.greenCreate(&p->gctx[p->n_gctx], desc, (CUdevice)p->dev, CU_GREEN_CTX_DEFAULT_STREAM));
        CKD(d.ctxFromGreen(&p->sctx[s], p->gctx[p->n_gctx]));
        p->n_gctx++;
        if (!lastst) {
            // the remainder must become a green context before it can be split again
            CUdevResourceDesc rdesc;
            CKD(d.genDesc(&rdesc, &rest, 1));
            CKD(d.greenCreate(&p->gctx[p->n_gctx], rdesc, (CUdevice)p->dev,
                              CU_GREEN_CTX_DEFAULT_STREAM));
            memset(&cur, 0, sizeof(cur));
            CKD(d.greenGetResource(p->gctx[p->n_gctx], &cur, CU_DEV_RESOURCE_TYPE_SM));
            p->n_gctx++;
        }
    }
    return SGP_OK;
}

}  // namespace

extern "C" int sgp_enumerate_splits(int n_sm, int quantum, int p_min, int* out, int max_out) {
    if (n_sm < 2 || quantum < 1 || p_min < 1) return fail_arg("n_sm, quantum, p_min");
    int lo = ((p_min + quantum - 1) / quantum) * quantum;
    int n = 0;
    for (int pa = lo; pa <= n_sm - p_min; pa += quantum) {
        if (out && n < max_out) out[n] = pa;
        ++n;
    }
    return n;
}

extern "C" int sgp_pipeline_create(const sgp_dims* d, const int* sm_split, int n_stages,
                                   int microbatch, int max_tokens, int max_kv_len,
                                   const sgp_pipeline_opts* opts, sgp_pipeline** out) {
    int r;
    if (!out) return fail_arg("out is NULL");
    *out = nullptr;
    if ((r = check_dims(d)) != SGP_OK) return r;
    if (n_stages < 1 || n_stages > 3) return fail_arg("n_stages must be 1, 2 or 3");
    if (microbatch < 1 || max_tokens < 1 || max_tokens % microbatch)
        return fail_arg("microbatch must divide max_tokens");
    if (max_tokens > kMaxTokens) return fail_arg("more than 512 sequences");
    if (d && d->rope_theta > 0.f && !use_tc_dense(*d, max_tokens))
        return fail_arg("RoPE needs the tensor-core QKV path");
    if (max_kv_len < 1) return fail_arg("max_kv_len");
    if (!drv().core) {
        g_err = "CUDA driver entry points unavailable";
        return SGP_ERR_UNSUPPORTED;
    }
    sgp_pipeline* p = new (std::nothrow) sgp_pipeline();
    if (!p) return SGP_ERR_OOM;
    p->dims = *d;
    p->n_stages = n_stages;
    p->micro = microbatch;
    p->max_tokens = max_tokens;
    p->max_kv = max_kv_len;
    if (opts)
        p->opts = *opts;
    else
        memset(&p->opts, 0, sizeof(p->opts));
    if (p->opts.custom_cut) {
        for (int s = 0; s < 2; ++s)
            for (int op = 0; op < SGP_N_OPS; ++op) {
                const int st = p->opts.stage_of_op[s][op];
                if (st < 0 || st >= n_stages) {
                    delete p;
                    return fail_arg("stage_of_op out of range");
                }
                p->stage_of_op[s][op] = st;
            }
    } else {
        for (int s = 0; s < 2; ++s)
            for (int op = 0; op < SGP_N_OPS; ++op) {
                int st = 0;
                if (n_stages == 2) st = op <= SGP_OP_ATTENTION ? 0 : 1;
                if (n_stages == 3)
                    st = op <= SGP_OP_ATTENTION ? 0 : (op <= SGP_OP_ROUTER ? 1 : 2);
                p->stage_of_op[s][op] = st;
            }
    }
    {
        const cudaError_t ge = cudaGetDevice(&p->dev);
        if (ge != cudaSuccess) {
            delete p;
            return fail_cuda(ge, "cudaGetDevice");
        }
    }
    const bool green = n_stages >= 2 && p->opts.use_green_contexts >= 0;
    if (green) {
        if (!sm_split) {
            delete p;
            return fail_arg("sm_split is NULL");
        }
        int nsm = 0;
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, p->dev);
        int sum = 0;
        for (int s = 0; s < n_stages; ++s) {
            if (sm_split[s] < 1) {
                delete p;
                return fail_arg("sm_split entries must be positive");
            }
            p->split[s] = sm_split[s];
            sum += sm_split[s];
        }
        if (sum > nsm) {
            delete p;
            return fail_arg("sm_split sums to more than the SM count");
        }
        if ((r = setup_green(p)) != SGP_OK) {
            sgp_pipeline_destroy(p);
            return r;
        }
    }
    if ((r = ensure_ws(p, max_tokens, 1)) != SGP_OK) {
        sgp_pipeline_destroy(p);
        return r;
    }
    cudaError_t ce = cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming);
    if (ce == cudaSuccess) ce = cudaHostAlloc((void**)&p->host_status, 16, cudaHostAllocDefault);
    if (ce != cudaSuccess) {
        sgp_pipeline_destroy(p);
        return fail_cuda(ce, "pipeline completion event / status copy");
    }
    memset(p->host_status, 0, 16);
    *out = p;
    return SGP_OK;
}

static int read_status(sgp_pipeline* p) {
    uint32_t st[4] = {0, 0, 0, 0};
    CK(cudaMemcpy(st, p->ws + p->lay.status, sizeof(st), cudaMemcpyDeviceToHost));
    if (p->host_status) p->host_status[0] = 0;
    if (st[0]) {
        CK(cudaMemset(p->ws + p->lay.status, 0, sizeof(st)));
        char buf[96];
        snprintf(buf, sizeof(buf), "device status 0x%x at op %u layer %u micro %u (detail %u)",
                 st[0], st[1] >> 24, (st[1] >> 12) & 0xFFF, st[1] & 0xFFF, st[2]);
        g_err = buf;
    }
    return status_to_code(st[0]);
}

static int pipeline_prepare(sgp_pipeline* p, const sgp_layer* layers, int n_layers,
                            const int32_t* kv_len, const void* x_in, void* x_out, int T) {
    int r;
    if (!p) return fail_arg("pipeline is NULL");
    if (!layers || n_layers < 1) return fail_arg("no layers");
    if (T < 1 || T > p->max_tokens || T % p->micro) return fail_arg("n_tokens vs microbatch");
    if (p->dims.rope_theta > 0.f && !use_tc_dense(p->dims, T))
        return fail_arg("RoPE needs the tensor-core QKV path");
    if (!kv_len || !x_in || !x_out || !aligned16(x_in) || !aligned16(x_out))
        return fail_arg("NULL or unaligned pointer");
    for (int l = 0; l < n_layers; ++l) {
        if ((r = check_layer(p->dims, &layers[l], T)) != SGP_OK) return r;
        if (layers[l].kv_cap > p->max_kv && layers[l].window == 0)
            return fail_arg("kv_cap above the pipeline's max_kv_len");
    }
    return SGP_OK;
}

extern "C" int sgp_pipeline_run(sgp_pipeline* p, const sgp_layer* layers, int n_layers,
                                const int32_t* kv_len, const void* x_in, void* x_out,
                                int n_tokens, int32_t* topk_idx, float* topk_w,
                                sgp_stream_t stream) {
    int r;
    if ((r = pipeline_prepare(p, layers, n_layers, kv_len, x_in, x_out, n_tokens)) != SGP_OK)
        return r;
    cudaStream_t s = (cudaStream_t)stream;
    if (p->launched) {
        // a device error of an earlier run that has completed: read from the pinned copy
        // that run left, without waiting for anything
        const cudaError_t q = cudaEventQuery(p->done);
        if (q == cudaSuccess) {
            if (p->host_status[0]) return read_status(p);
        } else if (q != cudaErrorNotReady) {
            return fail_cuda(q, "cudaEventQuery");
        }
        // the previous run (whatever stream it used) completes before this one starts: it
        // shares the pipeline's flags and scratch
        if (s != p->last_stream) CK(cudaStreamWaitEvent(s, p->done, 0));
    }
    std::vector<uint8_t> key;
    auto add = [&](const void* v, size_t n) {
        const uint8_t* b = (const uint8_t*)v;
        key.insert(key.end(), b, b + n);
    };
    add(layers, sizeof(sgp_layer) * n_layers);
    add(&kv_len, sizeof(kv_len));
    add(&x_in, sizeof(x_in));
    add(&x_out, sizeof(x_out));
    add(&n_tokens, sizeof(n_tokens));
    add(&topk_idx, sizeof(topk_idx));
    add(&topk_w, sizeof(topk_w));
    if (!p->exec || key != p->key) {
        // a rebuild may reallocate the scratch the previous run still uses: wait for it
        if (p->launched) CK(cudaEventSynchronize(p->done));
        const int m = n_tokens / p->micro;
        std::vector<PTask> tasks = build_tasks(*p, layers, n_layers, m);
        const int ntrace = p->opts.trace ? n_layers * m * SGP_N_OPS * 2 : 0;
        if ((r = ensure_ws(p, n_tokens, (int)tasks.size(), ntrace)) != SGP_OK) return r;
        // ensure_ws recomputed the layout for this token count
        if (p->lay.m != m) {
            cudaFree(p->ws);
            p->ws = nullptr;
            if ((r = ensure_ws(p, n_tokens, (int)tasks.size(), ntrace)) != SGP_OK) return r;
        }
        p->trace_pairs = ntrace;
        cudaGraph_t g;
        if ((r = build_graph(p, tasks, layers, kv_len, x_in, x_out, n_tokens, topk_idx, topk_w, -1,
                             &g)) != SGP_OK)
            return r;
        if (p->exec) {
            cudaGraphExecDestroy(p->exec);
            p->exec = nullptr;
        }
        cudaError_t e = cudaGraphInstantiate(&p->exec, g, 0);
        cudaGraphDestroy(g);
        if (e != cudaSuccess) return fail_cuda(e, "cudaGraphInstantiate");
        p->key = key;
        p->tasks = tasks;
    }
    CK(cudaGraphLaunch(p->exec, s));
    CK(cudaMemcpyAsync(p->host_status, p->ws + p->lay.status, 16, cudaMemcpyDeviceToHost, s));
    CK(cudaEventRecord(p->done, s));
    p->launched = true;
    p->last_stream = s;
    return SGP_OK;
}

extern "C" int sgp_pipeline_sync(sgp_pipeline* p) {
    if (!p) return fail_arg("pipeline is NULL");
    if (p->launched) CK(cudaEventSynchronize(p->done));
    return read_status(p);
}

namespace {
// Times each stage's tasks on its own pool (data edges between stages dropped), median of
// `reps` replays after one warm-up.  shared: all stages replay at the same time, each on its
// own stream, so every stage is timed while the others load HBM and L2 as in a pipelined
// run; otherwise one stage at a time, alone on the GPU.
int time_stages(sgp_pipeline* p, const std::vector<PTask>& tasks, const sgp_layer* layers,
                const int32_t* kv_len, const void* x_in, void* x_out, int T, int reps,
                bool shared, float* t_us) {
    const int n = p->n_stages;
    std::vector<cudaGraphExec_t> ex(n, nullptr);
    std::vector<cudaStream_t> st(n, nullptr);
    std::vector<cudaEvent_t> e0(n, nullptr), e1(n, nullptr);
    std::vector<std::vector<float>> ts(n);
    int r = SGP_OK;
    cudaError_t ce = cudaSuccess;
    for (int i = 0; i < n && r == SGP_OK && ce == cudaSuccess; ++i) {
        cudaGraph_t g;
        if ((r = build_graph(p, tasks, layers, kv_len, x_in, x_out, T, nullptr, nullptr, i, &g)) !=
            SGP_OK)
            break;
        ce = cudaGraphInstantiate(&ex[i], g, 0);
        cudaGraphDestroy(g);
        if (ce == cudaSuccess) ce = cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking);
        if (ce == cudaSuccess) ce = cudaEventCreate(&e0[i]);
        if (ce == cudaSuccess) ce = cudaEventCreate(&e1[i]);
    }
    for (int it = 0; it < reps + 1 && r == SGP_OK && ce == cudaSuccess; ++it) {
        for (int i = 0; i < n && ce == cudaSuccess; ++i) {
            ce = cudaEventRecord(e0[i], st[i]);
            if (ce == cudaSuccess) ce = cudaGraphLaunch(ex[i], st[i]);
            if (ce == cudaSuccess) ce = cudaEventRecord(e1[i], st[i]);
            if (ce == cudaSuccess && !shared) ce = cudaEventSynchronize(e1[i]);
        }
        for (int i = 0; i < n && ce == cudaSuccess; ++i) {
            ce = cudaEventSynchronize(e1[i]);
            float ms = 0.f;
            if (ce == cudaSuccess) ce = cudaEventElapsedTime(&ms, e0[i], e1[i]);
            if (ce == cudaSuccess && it > 0) ts[i].push_back(ms * 1000.f);
        }
    }
    for (int i = 0; i < n; ++i) {
        if (ex[i]) cudaGraphExecDestroy(ex[i]);
        if (e0[i]) cudaEventDestroy(e0[i]);
        if (e1[i]) cudaEventDestroy(e1[i]);
        if (st[i]) cudaStreamDestroy(st[i]);
    }
    if (r != SGP_OK) return r;
    if (ce != cudaSuccess) return fail_cuda(ce, "stage timing");
    for (int i = 0; i < n; ++i) {
        std::sort(ts[i].begin(), ts[i].end());
        t_us[i] = ts[i][ts[i].size() / 2];
    }
    return SGP_OK;
}
}  // namespace

extern "C" int sgp_pipeline_stage_times(sgp_pipeline* p, const sgp_layer* layers, int n_layers,
                                        const int32_t* kv_len, const void* x_in, void* x_out,
                                        int n_tokens, int reps, float* t_us) {
    int r;
    if ((r = pipeline_prepare(p, layers, n_layers, kv_len, x_in, x_out, n_tokens)) != SGP_OK)
        return r;
    if (!t_us || reps < 1) return fail_arg("t_us / reps");
    if (p->launched) CK(cudaEventSynchronize(p->done));  // the last run shares the scratch
    const int m = n_tokens / p->micro;
    std::vector<PTask> tasks = build_tasks(*p, layers, n_layers, m);
    if ((r = ensure_ws(p, n_tokens, (int)tasks.size())) != SGP_OK) return r;
    if (p->lay.m != m) {
        cudaFree(p->ws);
        p->ws = nullptr;
        if (p->exec) {
            cudaGraphExecDestroy(p->exec);
            p->exec = nullptr;
        }
        if ((r = ensure_ws(p, n_tokens, (int)tasks.size())) != SGP_OK) return r;
    }
    r = time_stages(p, tasks, layers, kv_len, x_in, x_out, n_tokens, reps,
                    p->opts.stage_times_shared != 0, t_us);
    if (r != SGP_OK) return r;
    return read_status(p);
}

extern "C" int sgp_pipeline_tasks(sgp_pipeline* p, int* n_tasks, int32_t* rows, int max_rows) {
    if (!p || !n_tasks) return fail_arg("NULL");
    *n_tasks = (int)p->tasks.size();
    if (rows)
        for (int i = 0; i < (int)p->tasks.size() && i < max_rows; ++i) {
            const PTask& t = p->tasks[i];
            rows[5 * i + 0] = t.stage;
            rows[5 * i + 1] = t.l0;
            rows[5 * i + 2] = t.mu;
            rows[5 * i + 3] = t.pred_data;
            rows[5 * i + 4] = t.pred_stage;
        }
    return SGP_OK;
}

extern "C" int sgp_pipeline_trace(sgp_pipeline* p, uint64_t* t_ns, int max_pairs, int* n_pairs) {
    if (!p || !n_pairs) return fail_arg("NULL");
    if (!p->opts.trace) return fail_arg("pipeline was created without opts.trace");
    if (!p->exec) return fail_arg("no run yet");
    *n_pairs = p->trace_pairs;
    if (!t_ns || max_pairs <= 0) return SGP_OK;
    if (p->launched) CK(cudaEventSynchronize(p->done));
    const int n = std::min(max_pairs, p->trace_pairs);
    std::vector<unsigned long long> h((size_t)n * 2);
    CK(cudaMemcpy(h.data(), p->ws + p->lay.trace, h.size() * 8, cudaMemcpyDeviceToHost));
    for (int i = 0; i < n; ++i) {
        t_ns[2 * i] = h[2 * i] ? ~h[2 * i] : 0;  // stored complemented (max of ~t = min t)
        t_ns[2 * i + 1] = h[2 * i + 1];
    }
    return SGP_OK;
}

extern "C" int sgp_pipeline_trace_sms(sgp_pipeline* p, uint32_t* masks, int max_entries,
                                      int* n_entries) {
    if (!p || !n_entries) return fail_arg("NULL");
    if (!p->opts.trace) return fail_arg("pipeline was created without opts.trace");
    if (!p->exec) return fail_arg("no run yet");
    *n_entries = p->trace_pairs;
    if (!masks || max_entries <= 0) return SGP_OK;
    if (p->launched) CK(cudaEventSynchronize(p->done));
    const int n = std::min(max_entries, p->trace_pairs);
    CK(cudaMemcpy(masks, p->ws + p->lay.smmask, (size_t)n * 32, cudaMemcpyDeviceToHost));
    return SGP_OK;
}

extern "C" int sgp_makespan(int n_tasks, const int32_t* pred_data, const int32_t* pred_stage,
                            const int32_t* stage, const double* tau, double handoff,
                            double* makespan, double* finish) {
    if (n_tasks < 0 || (n_tasks > 0 && (!pred_data || !pred_stage || !stage || !tau)) ||
        !makespan || !(handoff >= 0.0))
        return fail_arg("makespan arguments");
    std::vector<double> C((size_t)n_tasks, 0.0);
    double T = 0.0;
    for (int i = 0; i < n_tasks; ++i) {
        const int d = pred_data[i], q = pred_stage[i];
        if (d >= i || q >= i) return fail_arg("tasks are not in a topological order");
        double A = 0.0;
        if (d >= 0) A = std::max(A, C[d] + (stage[d] != stage[i] ? handoff : 0.0));
        if (q >= 0) A = std::max(A, C[q]);
        C[i] = A + tau[i];
        T = std::max(T, C[i]);
        if (finish) finish[i] = C[i];
    }
    *makespan = T;
    return SGP_OK;
}

namespace {
// Span {first-CTA start, last-CTA end} (ns) of every task, from a copy h of the launch trace
// ([layer][microbatch][op][part] pairs; the start is stored complemented).  {0, 0}: no launch.
void spans_from_trace(const std::vector<PTask>& tasks, int m,
                      const std::vector<unsigned long long>& h, std::vector<uint64_t>& spans) {
    spans.assign(tasks.size() * 2, 0);
    for (size_t i = 0; i < tasks.size(); ++i) {
        const PTask& t = tasks[i];
        uint64_t first = 0, last = 0;
        int l = t.l0, op = t.op0;
        while (true) {
            for (int part = 0; part < 2; ++part) {
                const size_t e = ((((size_t)l * m + t.mu) * SGP_N_OPS + op) * 2 + part) * 2;
                if (e + 1 >= h.size() || h[e + 1] == 0) continue;  // no such launch
                const uint64_t st = ~h[e], en = h[e + 1];
                if (first == 0 || st < first) first = st;
                if (en > last) last = en;
            }
            if (l == t.l1 && op == t.op1) break;
            if (++op == SGP_N_OPS) {
                op = 0;
                ++l;
            }
        }
        spans[2 * i] = first;
        spans[2 * i + 1] = last;
    }
}
}  // namespace

extern "C" int sgp_pipeline_task_spans(sgp_pipeline* p, uint64_t* spans, int max_tasks,
                                       int* n_tasks) {
    if (!p || !n_tasks) return fail_arg("NULL");
    if (!p->opts.trace) return fail_arg("pipeline was created without opts.trace");
    if (!p->exec) return fail_arg("no run yet");
    *n_tasks = (int)p->tasks.size();
    if (!spans || max_tasks <= 0) return SGP_OK;
    if (p->launched) CK(cudaEventSynchronize(p->done));
    std::vector<unsigned long long> h((size_t)p->trace_pairs * 2);
    CK(cudaMemcpy(h.data(), p->ws + p->lay.trace, h.size() * 8, cudaMemcpyDeviceToHost));
    std::vector<uint64_t> sp;
    spans_from_trace(p->tasks, p->lay.m, h, sp);
    for (int i = 0; i < (int)p->tasks.size() && i < max_tasks; ++i) {
        spans[2 * i] = sp[2 * i];
        spans[2 * i + 1] = sp[2 * i + 1];
    }
    return SGP_OK;
}

// Makespan of a run predicted by the pages' timing recurrence (Eq. 4-5) from task durations
// measured under contention: every stage replays its tasks at the same time, each on its own
// stream and pool, with the launch trace on; a task's duration tau_i runs from its start to
// the start of the next task of its FIFO (the last one: to its end), so it includes the gap
// a stage pays between tasks.  Then A_i = max(C_data + handoff (cross-stage), C_stage),
// C_i = A_i + tau_i, T = max C_i.
extern "C" int sgp_pipeline_predict(sgp_pipeline* p, const sgp_layer* layers, int n_layers,
                                    const int32_t* kv_len, const void* x_in, void* x_out,
                                    int n_tokens, float handoff_us, float* t_pred_us,
                                    float* t_stage_us) {
    int r;
    if ((r = pipeline_prepare(p, layers, n_layers, kv_len, x_in, x_out, n_tokens)) != SGP_OK)
        return r;
    if (!t_pred_us || !(handoff_us >= 0.f)) return fail_arg("t_pred_us / handoff_us");
    if (p->launched) CK(cudaEventSynchronize(p->done));  // the last run shares the scratch
    const int m = n_tokens / p->micro;
    std::vector<PTask> tasks = build_tasks(*p, layers, n_layers, m);
    const int ntrace = n_layers * m * SGP_N_OPS * 2;
    if (!p->ws || p->lay.m != m || p->ws_T != n_tokens || p->ws_nflags < (int)tasks.size() ||
        p->lay.n_trace < ntrace) {
        if (p->ws) {
            cudaFree(p->ws);
            p->ws = nullptr;
        }
        if (p->exec) {
            cudaGraphExecDestroy(p->exec);
            p->exec = nullptr;
        }
        if ((r = ensure_ws(p, n_tokens, (int)tasks.size(), ntrace)) != SGP_OK) return r;
    }
    const int n = p->n_stages;
    std::vector<cudaGraphExec_t> ex(n, nullptr);
    std::vector<cudaStream_t> st(n, nullptr);
    cudaEvent_t ev = nullptr;
    cudaError_t ce = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    for (int i = 0; i < n && r == SGP_OK && ce == cudaSuccess; ++i) {
        cudaGraph_t g;
        if ((r = build_graph(p, tasks, layers, kv_len, x_in, x_out, n_tokens, nullptr, nullptr, i,
                             &g, false)) != SGP_OK)
            break;
        ce = cudaGraphInstantiate(&ex[i], g, 0);
        cudaGraphDestroy(g);
        if (ce == cudaSuccess) ce = cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking);
    }
    // two replays (the first warms up), each after one clear of counters, flags and trace
    for (int rep = 0; rep < 2 && r == SGP_OK && ce == cudaSuccess; ++rep) {
        ce = cudaMemsetAsync(p->ws + p->lay.zero_beg, 0, p->lay.zero_end - p->lay.zero_beg, st[0]);
        if (ce == cudaSuccess) ce = cudaEventRecord(ev, st[0]);
        for (int i = 0; i < n && ce == cudaSuccess; ++i) {
            if (i > 0) ce = cudaStreamWaitEvent(st[i], ev, 0);
            if (ce == cudaSuccess) ce = cudaGraphLaunch(ex[i], st[i]);
        }
        for (int i = 0; i < n && ce == cudaSuccess; ++i) ce = cudaStreamSynchronize(st[i]);
    }
    std::vector<unsigned long long> h((size_t)ntrace * 2);
    if (r == SGP_OK && ce == cudaSuccess)
        ce = cudaMemcpy(h.data(), p->ws + p->lay.trace, h.size() * 8, cudaMemcpyDeviceToHost);
    for (int i = 0; i < n; ++i) {
        if (ex[i]) cudaGraphExecDestroy(ex[i]);
        if (st[i]) cudaStreamDestroy(st[i]);
    }
    if (ev) cudaEventDestroy(ev);
    if (r != SGP_OK) return r;
    if (ce != cudaSuccess) return fail_cuda(ce, "prediction replay");
    std::vector<uint64_t> sp;
    spans_from_trace(tasks, m, h, sp);
    // durations: start to the next start on the same FIFO (stage and lane)
    const int lanes = p->opts.stage_lanes == 2 ? 2 : 1;
    std::vector<double> tau(tasks.size(), 0.0);
    std::vector<int> next(tasks.size(), -1);
    int last_on[4][2] = {{-1, -1}, {-1, -1}, {-1, -1}, {-1, -1}};
    for (size_t i = 0; i < tasks.size(); ++i) {
        int& prev = last_on[tasks[i].stage][tasks[i].mu % lanes];
        if (prev >= 0) next[prev] = (int)i;
        prev = (int)i;
    }
    double t_st[4] = {0, 0, 0, 0};
    for (size_t i = 0; i < tasks.size(); ++i) {
        const double s0 = (double)sp[2 * i], e0 = (double)sp[2 * i + 1];
        if (e0 == 0) continue;  // a task with no launch takes no time
        double t = e0 - s0;
        if (next[i] >= 0 && sp[2 * next[i] + 1] != 0) t = std::max(t, (double)sp[2 * next[i]] - s0);
        tau[i] = t * 1e-3;
        t_st[tasks[i].stage] += tau[i];
    }
    std::vector<int32_t> pd(tasks.size()), ps(tasks.size()), stg(tasks.size());
    for (size_t i = 0; i < tasks.size(); ++i) {
        pd[i] = tasks[i].pred_data;
        ps[i] = tasks[i].pred_stage;
        stg[i] = tasks[i].stage;
    }
    double T = 0.0;
    if ((r = sgp_makespan((int)tasks.size(), pd.data(), ps.data(), stg.data(), tau.data(),
                          handoff_us, &T, nullptr)) != SGP_OK)
        return r;
    *t_pred_us = (float)T;
    if (t_stage_us)
        for (int i = 0; i < n; ++i) t_stage_us[i] = (float)t_st[i];
    return read_status(p);
}

extern "C" void sgp_pipeline_destroy(sgp_pipeline* p) {
    if (!p) return;
    if (p->launched) cudaEventSynchronize(p->done);
    if (p->exec) cudaGraphExecDestroy(p->exec);
    if (p->ws) cudaFree(p->ws);
    if (p->done) cudaEventDestroy(p->done);
    if (p->host_status) cudaFreeHost(p->host_status);
    Driver& d = drv();
    for (int i = p->n_gctx - 1; i >= 0; --i)
        if (p->gctx[i] && d.greenDestroy) d.greenDestroy(p->gctx[i]);
    delete p;
}

// =======================================================================================
// C ABI: pairwise-line SM-allocation refinement ("SubGPU Pipelining", Section 4.2,
// Algorithm 2).  A move p^{d->r}[z] hands z quanta of SMs from donor stage d to receiver
// stage r.  Each pass takes the best one-quantum move; if it improves the objective, a
// doubling/halving line search extends it along the same (d, r) pair.  Objective values
// are memoised per allocation.
// =======================================================================================
namespace {
struct AllocSearch {
    int n;
    int g, p_min;
    sgp_alloc_objective f;
    void* ctx;
    std::vector<std::pair<std::vector<int>, double>> memo;
    int evals = 0;
    bool feasible(const std::vector<int>& p) const {
        for (int v : p)
            if (v < p_min || v < g) return false;
        return true;
    }
    // objective, memoised; an allocation the objective cannot evaluate (< 0) is +inf
    double eval(const std::vector<int>& p) {
        for (const auto& e : memo)
            if (e.first == p) return e.second;
        double t = f(p.data(), n, ctx);
        ++evals;
        if (!(t >= 0.0)) t = INFINITY;
        memo.emplace_back(p, t);
        return t;
    }
    std::vector<int> moved(const std::vector<int>& p, int d, int r, int z) const {
        std::vector<int> q = p;
        q[d] -= z * g;
        q[r] += z * g;
        return q;
    }
};
}  // namespace

extern "C" int sgp_refine_allocation(int n_stages, int* p_inout, int quantum, int p_min,
                                     int pass_limit, sgp_alloc_objective f, void* ctx,
                                     double* t_out) {
    if (n_stages < 2 || n_stages > 8 || !p_inout || quantum < 1 || p_min < 0 || !f)
        return fail_arg("n_stages, p, quantum, p_min or objective");
    AllocSearch S{n_stages, quantum, p_min, f, ctx, {}, 0};
    std::vector<int> p(p_inout, p_inout + n_stages);
    if (!S.feasible(p)) return fail_arg("initial allocation below p_min or the quantum");
    double t = S.eval(p);
    for (int pass = 1; pass_limit <= 0 || pass <= pass_limit; ++pass) {
        int bd = -1, br = -1;
        double t_line = INFINITY;
        for (int d = 0; d < n_stages; ++d)
            for (int r = 0; r < n_stages; ++r) {
                if (d == r) continue;
                const std::vector<int> q = S.moved(p, d, r, 1);
                if (!S.feasible(q)) continue;
                const double v = S.eval(q);
                if (bd < 0 || v < t_line) {  // first minimum in (d, r) order
                    bd = d;
                    br = r;
                    t_line = v;
                }
            }
        if (bd < 0 || !(t_line < t)) break;  // no legal move, or none improves
        int z = 1, h = 1;
        while (h > 0) {
            const std::vector<int> q = S.moved(p, bd, br, z + h);
            double v;
            if (S.feasible(q) && (v = S.eval(q)) < t_line) {
                z += h;
                t_line = v;
                h *= 2;
            } else {
                h /= 2;
            }
        }
        p = S.moved(p, bd, br, z);
        t = t_line;
    }
    for (int i = 0; i < n_stages; ++i) p_inout[i] = p[i];
    if (t_out) *t_out = t;
    return S.evals;
}

namespace {
struct RefineCtx {
    const sgp_dims* d;
    const sgp_layer* layers;
    int n_layers;
    const int32_t* kv_len;
    const void* x_in;
    void* x_out;
    int T, micro, max_kv, reps;
    const sgp_pipeline_opts* opts;
    int err = SGP_OK;  // first error other than an allocation the device cannot form
};

// objective: the median time (us) of `reps` full pipelined runs with SM allocation p
double refine_objective(const int* split, int n, void* vctx) {
    RefineCtx& c = *static_cast<RefineCtx*>(vctx);
    if (c.err != SGP_OK) return -1.0;
    sgp_pipeline* p = nullptr;
    int r = sgp_pipeline_create(c.d, split, n, c.micro, c.T, c.max_kv, c.opts, &p);
    if (r != SGP_OK) return -1.0;  // a split the device cannot form is infeasible
    cudaStream_t s = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    std::vector<float> ts;
    cudaError_t ce = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (ce == cudaSuccess) ce = cudaEventCreate(&e0);
    if (ce == cudaSuccess) ce = cudaEventCreate(&e1);
    for (int i = 0; i < c.reps + 1 && ce == cudaSuccess && r == SGP_OK; ++i) {
        ce = cudaEventRecord(e0, s);
        if (ce != cudaSuccess) break;
        r = sgp_pipeline_run(p, c.layers, c.n_layers, c.kv_len, c.x_in, c.x_out, c.T, nullptr,
                             nullptr, s);
        if (r != SGP_OK) break;
        ce = cudaEventRecord(e1, s);
        if (ce == cudaSuccess) ce = cudaEventSynchronize(e1);
        float ms = 0.f;
        if (ce == cudaSuccess) ce = cudaEventElapsedTime(&ms, e0, e1);
        if (ce == cudaSuccess && i > 0) ts.push_back(ms * 1000.f);
    }
    if (r == SGP_OK && ce == cudaSuccess) r = sgp_pipeline_sync(p);
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    if (s) cudaStreamDestroy(s);
    sgp_pipeline_destroy(p);
    if (ce != cudaSuccess) r = fail_cuda(ce, "refinement run");
    if (r != SGP_OK) {
        c.err = r;
        return -1.0;
    }
    std::sort(ts.begin(), ts.end());
    return ts[ts.size() / 2];
}
}  // namespace

extern "C" int sgp_pipeline_refine(const sgp_dims* d, const sgp_layer* layers, int n_layers,
                                   const int32_t* kv_len, const void* x_in, void* x_out,
                                   int n_tokens, int n_stages, int microbatch, int max_kv_len,
                                   int quantum, int reps, int pass_limit,
                                   const sgp_pipeline_opts* opts, int* split_inout,
                                   float* t_us_out, int* n_evals) {
    if (!split_inout || reps < 1 || n_stages < 2 || n_stages > 3)
        return fail_arg("split, reps or n_stages (2 or 3)");
    sgp_device_info info;
    int r;
    if ((r = sgp_device_info_get(&info)) != SGP_OK) return r;
    if (!info.green_ctx_supported) return SGP_ERR_UNSUPPORTED;
    const int q = std::max(quantum, std::max(1, info.sm_alignment));
    const int pmin = std::max(q, info.sm_min_partition);
    RefineCtx c{d, layers, n_layers, kv_len, x_in, x_out, n_tokens, microbatch, max_kv_len, reps,
                opts};
    double t = 0.0;
    const int ev = sgp_refine_allocation(n_stages, split_inout, q, pmin, pass_limit,
                                         refine_objective, &c, &t);
    if (ev < 0) return ev;
    if (c.err != SGP_OK) return c.err;
    if (!std::isfinite(t)) return fail_arg("no allocation could be run");
    if (t_us_out) *t_us_out = (float)t;
    if (n_evals) *n_evals = ev;
    return SGP_OK;
}

extern "C" int sgp_pipeline_balance(const sgp_dims* d, const sgp_layer* layers, int n_layers,
                                    const int32_t* kv_len, const void* x_in, void* x_out,
                                    int n_tokens, int microbatch, int max_kv_len, int quantum,
                                    int reps, const sgp_pipeline_opts* opts, int* best_split_out,
                                    int* splits, float* t_us, int max_out, int* n_out) {
    int r;
    if (!best_split_out || !n_out) return fail_arg("NULL output");
    sgp_device_info info;
    if ((r = sgp_device_info_get(&info)) != SGP_OK) return r;
    if (!info.green_ctx_supported) return SGP_ERR_UNSUPPORTED;
    const int q = std::max(quantum, std::max(1, info.sm_alignment));
    const int pmin = std::max(q, info.sm_min_partition);
    std::vector<int> cand(sgp_enumerate_splits(info.sm_count, q, pmin, nullptr, 0));
    sgp_enumerate_splits(info.sm_count, q, pmin, cand.data(), (int)cand.size());
    float best = INFINITY;
    *best_split_out = -1;
    int n = 0;
    for (int pa : cand) {
        int split[2] = {pa, info.sm_count - pa};
        sgp_pipeline* p = nullptr;
        if ((r = sgp_pipeline_create(d, split, 2, microbatch, n_tokens, max_kv_len, opts, &p)) !=
            SGP_OK)
            continue;  // a split the device cannot form is skipped
        float t[2] = {0.f, 0.f};
        r = sgp_pipeline_stage_times(p, layers, n_layers, kv_len, x_in, x_out, n_tokens, reps, t);
        sgp_pipeline_destroy(p);
        if (r != SGP_OK) return r;
        if (n < max_out) {
            if (splits) splits[n] = pa;
            if (t_us) {
                t_us[2 * n] = t[0];
                t_us[2 * n + 1] = t[1];
            }
        }
        ++n;
        const float mx = std::max(t[0], t[1]);
        if (mx < best) {
            best = mx;
            *best_split_out = pa;
        }
    }
    *n_out = n;
    return *best_split_out >= 0 ? SGP_OK : SGP_ERR_UNSUPPORTED;
}
