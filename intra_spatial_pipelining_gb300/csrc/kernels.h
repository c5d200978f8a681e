// Problem descriptions of the layer's kernels and the host-side enqueue functions.
// Each kernel translation unit owns its kernels; the runtime only sees these functions,
// which compute the launch shape and hand the launch to a Launcher (a stream, or a CUDA
// graph under construction bound to one SM pool).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace sgp {

// Receives launches.  args points to one pointer per kernel parameter (cudaLaunchKernel
// convention); the launcher copies the values before returning.  Returns a cudaError_t.
struct Launcher {
    virtual ~Launcher() {}
    // overlap_ok: the kernel may be launched programmatically after its predecessor (it only
    // touches memory the predecessor writes after griddep_wait)
    virtual int launch(const void* func, dim3 grid, dim3 block, size_t smem, void** args,
                       bool overlap_ok = false) = 0;
    // A launch beside the chain: it starts once the chain's last launch so far has completed,
    // and nothing in the chain waits for it.  For work whose effect is only on timing (an L2
    // prefetch); a launcher without side branches drops it.
    virtual int launch_side(const void* func, dim3 grid, dim3 block, size_t smem, void** args) {
        (void)func, (void)grid, (void)block, (void)smem, (void)args;
        return 0;
    }
};

// --------------------------------------------------------------------------------------
// projection epilogues
// --------------------------------------------------------------------------------------
enum EpiMode : int { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_F32 = 3 };

struct EpiArgs {
    int mode;
    int n_out;          // valid output features (per group)
    int ld;             // row stride (elements) of the output / residual rows
    // EPI_QKV: q [rows][q_width]; caches [seq][nkv][cap][d]
    bf16* q;
    int q_width;
    bf16* kc;
    bf16* vc;
    const int* kv_len;
    int nkv, cap, d;
    float rope_theta;       // EPI_QKV: RoPE base for q and k (0: none)
    float rope_fhi[32], rope_flo[32];  // theta^(-2i/64) as hi + lo float pairs (host, in double)
    // EPI_RESID: out = resid + acc (bf16); EPI_SWIGLU: out = silu(gate) * up (bf16)
    const bf16* resid;
    bf16* out;
    // EPI_F32
    float* out_f32;
};

// Skinny GEMM  D[out_feature][token] = sum_k W[out_feature][k] * X[token][k]  on tcgen05.
// Work unit = (group, 128-row tile, K segment); the K split is fixed by the shape so the
// fp32 summation order never depends on the grid or on the token count.
// Each pipeline stage holds kps (1 or 2) consecutive 64-wide k-blocks: the 128-row weight
// tile arrives in ONE TMA operation (16 or 32 KB) and the stage's activation rows in one
// more.  Two k-blocks per stage when a pass carries few tokens (larger weight boxes stream
// faster); one when it carries many, so that the ring stays deep although the activation
// rows dominate the stage.
constexpr int kGemmKpsMax = 2;
// tokens per pass go up to 256 (one MMA's N); the accumulator is drained through shared
// memory kTsRows tokens at a time
constexpr int kGemmMaxN = 256;
constexpr int kTsRows = 64;
// shared memory of one projection CTA (ring + staging + barriers): well under the SM's
// 228 KB, so that a small kernel's CTA fits beside it
constexpr int kGemmSmemBudget = 200 * 1024;
// a grouped (expert) projection's kernel before it needs only a few KB of shared memory
constexpr int kGemmSmemBudgetGrouped = 221 * 1024;

struct GemmProblem {
    // weights: plain  3-D {64, rows, k-blocks} box {64, 128, 2};
    //          SwiGLU 4-D {64, rows, half, k-blocks} box {64, 64, 2, 2}, half = gate/up (I rows)
    CUtensorMap tmA;
    CUtensorMap tmB;        // activations, 3-D {64, rows, k-blocks}, box {64, n_cap, 2}, SW128
    CUtensorMap tmB2;       // the same activations, box {64, tail_cap, kps} (tail_cap > 0)
    int a_4d;               // 1: SwiGLU (4-D weight map)
    int K, kb_total, ksplit;
    int kps;                // k-blocks per stage (1 or 2)
    int n_sb;               // stage blocks = ceil(kb_total / kps); K segments split these
    int m_tiles;            // 128-row tiles per group
    int n_groups;
    int rows_per_group;     // weight rows of one group
    int a_tile_stride;      // first weight row of tile mt = mt * a_tile_stride (128 or 64)
    int a_second_off;       // second 64-row half starts a_second_off rows later (64 or inter)
    const int* group_offsets;  // device [n_groups + 1] token-row ranges, or NULL (dense)
    int row0, nrows;        // dense: token rows [row0, row0 + nrows)
    int R;                  // rows of the partial-sum buffer
    int n_cap;              // tokens per pass (multiple of 16, <= kGemmMaxN)
    int tail_cap;           // grouped only: a last pass of at most tail_cap rows joins the pass
                            //    before it (a second accumulator fed by its own rows in every
                            //    stage), so the weight tile is not streamed once more for a few
                            //    rows; 0 = off.  Multiple of 16.
    int ts_rows;            // tokens per chunk of the accumulator's way out through shared memory
    int stages;             // shared-memory pipeline depth
    int ring_bytes;         // bytes of the stage ring (also holds the staged accumulator)
    int serpentine;         // visit groups in reverse order
    int keep_weights;       // 1: weight loads hint L2 evict-last (a later microbatch rereads
                            //    them), 0: evict-first
    float* partial;         // [m_tiles][ksplit][R][128] fp32 tiles (token-major rows)
    int n_units;            // n_groups * m_tiles * ksplit
    int grid;               // persistent CTAs (one per SM of the pool)
    // ksplit == 1: the epilogue is applied here from the staged tile (no partials, no
    // finishing pass); out_row0 = output row of partial row 0
    int fused_epi;
    int out_row0;
    EpiArgs epi;
};

// Sum of the K segments of every partial tile + fused epilogue.
struct FinishProblem {
    const float* partial;   // as GemmProblem::partial
    int ksplit, m_tiles, R;
    int rows;               // partial rows to finish: [0, rows)
    int out_row0;           // output row of partial row 0
    EpiArgs epi;
};

// Same contraction on CUDA cores (small token counts).
struct GemvProblem {
    const bf16* W;          // [groups * rows_per_group][K]
    int K, rows_per_group, n_groups, n_out, swiglu, up_off;
    const bf16* X;          // activations [rows][K]
    const int* group_offsets;
    int row0, nrows;
    EpiArgs epi;
};

struct AttnProblem {
    CUtensorMap tmK, tmV;   // caches as 2-D [seq * nkv * cap][64], box {64, pos}, SW128
    const bf16* q;          // [T][nq * 64]
    const int* kv_len;      // [T]
    bf16* o;                // [T][nq * 64]
    float* part_ml;         // [nrows * nkv][S_max][16 heads][2]  (max, sum)
    float* part_acc;        // [nrows * nkv][S_max][64 dims][16 heads]
    uint32_t* cnt;          // [nrows * nkv]
    int row0, nrows, nq, nkv, G, cap, window, chunk, S_max;
    float scale_log2;       // log2(e) / sqrt(d)
    int n_cta;              // persistent CTAs (one per SM of the pool)
    int pos;                // positions per stage (64 or 128; the K / V box height)
    // 1: the K and V halves of a stage are waited on and refilled separately (K after the
    // scores, V after the V product); 0: together, after the V product.  Load schedule only:
    // the results are identical either way.
    int kv_split;
};

struct NormProblem {
    const bf16* x;
    const bf16* g;
    bf16* y;
    int row0, nrows, H;
    float eps;
};

struct RouterProblem {
    const bf16* h;          // [T][H] batch-wide
    const bf16* g;          // [H]
    bf16* u;                // [T][H] batch-wide
    const bf16* Wr;         // [E][H]
    const float* bias;      // [E] or NULL
    float* logits;          // [nrows][E]
    int* idx;               // [nrows][k]
    float* wts;             // [nrows][k]
    int* user_idx;          // [T][k] batch-wide or NULL
    float* user_w;
    uint32_t* cnt;          // [ceil(nrows / 8)]
    int row0, nrows, H, E, k;
    float eps;
};

struct DispatchProblem {
    const int* idx;         // [nrows][k]
    const bf16* u;          // [T][H] batch-wide
    bf16* xperm;            // [nrows * k][H]
    int* offsets;           // [E_local + 1]
    int* pair_pos;          // [nrows * k]
    int row0, nrows, k, H, E, E_local, slot_map;
};

struct CombineProblem {
    const bf16* h;          // [T][H] batch-wide
    // expert-down output: ksplit == 1: rows [nrows * k][H]; ksplit > 1: the projection's K
    // segments, [H / 128][ksplit][R][128] (summed here in segment order)
    const float* Y;
    int ksplit, R;
    const float* wts;       // [nrows][k]
    const int* pair_pos;    // [nrows * k]
    bf16* out;              // [T][H] batch-wide
    int row0, nrows, k, H;
    // optional: the next layer's a = RMSNorm(out; g_next) in the same pass (H <= 4096)
    const bf16* g_next;     // or NULL
    bf16* a_next;           // [T][H] batch-wide
    float eps;
};

// L2 prefetch of up to two byte ranges (16-byte aligned, multiples of 16 bytes), with an
// evict-last hint so that the lines stay until the projection that reads them.
struct PrefetchProblem {
    const void* base[2];
    size_t bytes[2];
    int grid;               // CTAs (one warp each), spread over the pool's SMs
};

// Virtual communication: copy `bytes` (a multiple of 16) from src to dst, lasting at least
// floor_ns from the moment the payload is ready.
struct CommProblem {
    const void* src;
    void* dst;
    size_t bytes;
    unsigned long long floor_ns;
};

// --------------------------------------------------------------------------------------
// host enqueue functions (return cudaError_t as int)
// --------------------------------------------------------------------------------------
int enqueue_rmsnorm(Launcher& L, const NormProblem& p, const KCtx& c);
int enqueue_comm(Launcher& L, const CommProblem& p, const KCtx& c);
int enqueue_prefetch(Launcher& L, const PrefetchProblem& p, const KCtx& c);
int enqueue_router(Launcher& L, const RouterProblem& p, const KCtx& c);
int enqueue_dispatch(Launcher& L, const DispatchProblem& p, const KCtx& c);
int enqueue_combine(Launcher& L, const CombineProblem& p, const KCtx& c);
int enqueue_attention(Launcher& L, const AttnProblem& p, const KCtx& c);
int enqueue_gemm_tc(Launcher& L, const GemmProblem& p, const KCtx& c);
int enqueue_gemm_finish(Launcher& L, const FinishProblem& p, const KCtx& c);
int enqueue_gemv(Launcher& L, const GemvProblem& p, const KCtx& c);

// shared-memory bytes a tcgen05 GEMM launch needs for (n_cap, stages)
size_t gemm_tc_ring_bytes(int n_cap, int stages, int kps, int tail_cap, int ts_rows);
size_t gemm_tc_smem_bytes(int n_cap, int stages, int kps, int tail_cap, int ts_rows);
// attention chunk length (positions per split-KV work item); fixed, never SM-dependent
constexpr int kAttnChunk = 1024;
// Positions per attention stage for a call: 64 (12 warps per CTA) when the full batch has at
// least 8192 split-KV chunks, else 128 (6 warps).  A function of the shape alone, never of
// the SM pool, since it fixes the order of the fp32 online softmax.
inline int attn_stage_pos(long long n_chunks) { return n_chunks >= 8192 ? 64 : 128; }

}  // namespace sgp
