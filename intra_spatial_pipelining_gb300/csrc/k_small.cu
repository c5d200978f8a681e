// The latency-bound kernels of the layer: RMSNorm, router (RMSNorm + logits + top-k),
// dispatch (stable counting sort of the routed pairs by expert slot + row gather) and the
// weighted combine with the residual.  All loads and stores are 16-byte vectors, every
// reduction has a fixed order, and each token's result depends only on that token.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "sgp.h"

namespace sgp {

namespace {

// ---------------------------------------------------------------------------------------
// RMSNorm: y = bf16(x * rsqrt(mean(x^2) + eps) * g), one CTA per row
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rmsnorm_kernel(const NormProblem P, const KCtx ctx) {
    griddep_launch();
    griddep_wait();
    task_begin(ctx);
    __shared__ float red[8];
    const int row = P.row0 + blockIdx.x;
    const int nv = P.H >> 3;
    const uint4* x = reinterpret_cast<const uint4*>(P.x + (size_t)row * P.H);
    const uint4* g = reinterpret_cast<const uint4*>(P.g);
    uint4* y = reinterpret_cast<uint4*>(P.y + (size_t)row * P.H);
    float ss = 0.f;
    for (int v = threadIdx.x; v < nv; v += 256) {
        float f[8];
        unpack8(x[v], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float inv = rsqrtf(tot / (float)P.H + P.eps);
    for (int v = threadIdx.x; v < nv; v += 256) {
        float f[8], gg[8];
        unpack8(x[v], f);
        unpack8(g[v], gg);
        uint4 o;
        o.x = pack_bf16x2(f[0] * inv * gg[0], f[1] * inv * gg[1]);
        o.y = pack_bf16x2(f[2] * inv * gg[2], f[3] * inv * gg[3]);
        o.z = pack_bf16x2(f[4] * inv * gg[4], f[5] * inv * gg[5]);
        o.w = pack_bf16x2(f[6] * inv * gg[6], f[7] * inv * gg[7]);
        y[v] = o;
    }
    task_end(ctx);
}

// ---------------------------------------------------------------------------------------
// Router.  grid = (token groups of 16, expert groups of 8), 16 warps.
//   (0) the CTA's 8 router rows and the gain g go to shared memory by cp.async;
//   (1) warp w normalises token w: u = bf16(RMSNorm(h; g)) into shared memory (rows padded
//       by 16 bytes so ldmatrix rows fall on distinct banks) and, from the first expert
//       group, to global memory;
//   (2) logits z = u W_r^T on warp-level bf16 tensor-core MMAs with fp32 accumulation
//       (M = 16 tokens, N = 8 experts, two N tiles per CTA); the 16 warps split K and their
//       partial tiles are added in warp order;
//   (3) the last CTA of a token group selects each token's top-k (descending logit, ties to
//       the lower index, a NaN logit ranks below every number) and the softmax over the
//       selected logits, one warp per token.
// ---------------------------------------------------------------------------------------
constexpr int kRouterTok = 16;
constexpr int kRouterWarps = 16;
// experts per CTA: 16 (two 8-wide MMA tiles) where the rows fit in shared memory, else 8

__host__ __device__ inline int router_row_bytes(int H) { return H * 2 + 16; }
// u rows, router rows and g (the first two reused for the logit rows of the top-k), then the
// MMA partials
__host__ __device__ inline size_t router_rows_bytes(int H, int E, int NE) {
    const size_t rows = (size_t)(kRouterTok + NE + 1) * router_row_bytes(H);
    const size_t logit_rows = (size_t)kRouterWarps * E * sizeof(float);
    return rows > logit_rows ? rows : logit_rows;
}
inline size_t router_smem_bytes(int H, int E, int NE) {
    return router_rows_bytes(H, E, NE) + (size_t)kRouterWarps * 16 * NE * sizeof(float);
}
// experts per CTA: 16 for many tokens (half the CTAs, half the repeated RMSNorm work) when
// that fits the opt-in shared memory (with margin); 8 for few tokens (more CTAs in flight).
// Both give the same logits: every expert's dot product is split over the warps alike.
inline int router_experts_per_cta(int H, int E, int nrows) {
    return nrows >= 128 && router_smem_bytes(H, E, 16) <= 220 * 1024 ? 16 : 8;
}

__device__ __forceinline__ void ldsm_x4_r(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_r(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}

template <int NE>
__global__ void __launch_bounds__(kRouterWarps * 32, 1)
    router_kernel(const RouterProblem P, const KCtx ctx) {
    constexpr int kRouterExp = NE;
    griddep_launch();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int rb = router_row_bytes(P.H);
    uint8_t* u_s = smem_raw;                                   // [16][rb]
    uint8_t* w_s = u_s + (size_t)kRouterTok * rb;              // [kRouterExp][rb]
    uint8_t* g_s = w_s + (size_t)kRouterExp * rb;              // [rb]
    float* red = reinterpret_cast<float*>(smem_raw + router_rows_bytes(P.H, P.E, NE));  // [16][16][NE]
    __shared__ int sh_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tg = blockIdx.x;
    const int nv = P.H >> 3;
    const int ntok = min(kRouterTok, P.nrows - tg * kRouterTok);
    const int e0 = blockIdx.y * kRouterExp;
    const uint4 z4 = make_uint4(0, 0, 0, 0);

    // (0) router rows of experts e0 .. e0+NE-1 (rows past E are zero) and g, by cp.async: layer
    // constants, so they are requested before the previous kernel has finished
    static_assert(NE == 8 || NE == 16, "one or two 8-wide tiles");
    if (warp < NE) {
        const int e = e0 + warp;
        uint8_t* dst = w_s + (size_t)warp * rb;
        if (e < P.E) {
            const uint4* src = reinterpret_cast<const uint4*>(P.Wr + (size_t)e * P.H);
            for (int v = lane; v < nv; v += 32) cp_async16(dst + v * 16, src + v);
        } else {
            for (int v = lane; v < nv; v += 32) *reinterpret_cast<uint4*>(dst + v * 16) = z4;
        }
    }
    {
        const uint4* gsrc = reinterpret_cast<const uint4*>(P.g);
        for (int v = threadIdx.x; v < nv; v += kRouterWarps * 32) cp_async16(g_s + v * 16, gsrc + v);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    griddep_wait();
    task_begin(ctx);

    // (1) u = RMSNorm(h; g) of token `warp` (rows past the group are zero)
    constexpr int kRV = 12;  // 16-byte vectors per lane kept in registers (H <= 3072)
    const bool has_t = warp < ntok;
    const int row = P.row0 + tg * kRouterTok + (has_t ? warp : 0);
    const uint4* hrow = reinterpret_cast<const uint4*>(P.h + (size_t)row * P.H);
    uint4* uo = reinterpret_cast<uint4*>(P.u + (size_t)row * P.H);
    uint8_t* udst = u_s + (size_t)warp * rb;
    const uint4* gs4 = reinterpret_cast<const uint4*>(g_s);
    auto put = [&](int v, const uint4& hq, float inv) {
        float f[8], gg[8];
        unpack8(hq, f);
        unpack8(gs4[v], gg);
        uint4 o;
        o.x = pack_bf16x2(f[0] * inv * gg[0], f[1] * inv * gg[1]);
        o.y = pack_bf16x2(f[2] * inv * gg[2], f[3] * inv * gg[3]);
        o.z = pack_bf16x2(f[4] * inv * gg[4], f[5] * inv * gg[5]);
        o.w = pack_bf16x2(f[6] * inv * gg[6], f[7] * inv * gg[7]);
        *reinterpret_cast<uint4*>(udst + v * 16) = o;
        if (blockIdx.y == 0) uo[v] = o;
    };
    if (nv <= 32 * kRV) {
        uint4 hv[kRV];
#pragma unroll
        for (int i = 0; i < kRV; ++i) {
            const int v = i * 32 + lane;
            hv[i] = (has_t && v < nv) ? hrow[v] : z4;
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < kRV; ++i) {
            float f[8];
            unpack8(hv[i], f);
#pragma unroll
            for (int q = 0; q < 8; ++q) ss = fmaf(f[q], f[q], ss);
        }
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss / (float)P.H + P.eps);
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();  // g (and the router rows) visible to every warp
        if (has_t) {
#pragma unroll
            for (int i = 0; i < kRV; ++i) {
                const int v = i * 32 + lane;
                if (v < nv) put(v, hv[i], inv);
            }
        } else {
            for (int v = lane; v < nv; v += 32) *reinterpret_cast<uint4*>(udst + v * 16) = z4;
        }
    } else {
        float ss = 0.f;
        if (has_t)
            for (int v = lane; v < nv; v += 32) {
                float f[8];
                unpack8(hrow[v], f);
#pragma unroll
                for (int q = 0; q < 8; ++q) ss = fmaf(f[q], f[q], ss);
            }
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss / (float)P.H + P.eps);
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        if (has_t) {
            for (int v = lane; v < nv; v += 32) put(v, hrow[v], inv);
        } else {
            for (int v = lane; v < nv; v += 32) *reinterpret_cast<uint4*>(udst + v * 16) = z4;
        }
    }
    __syncthreads();

    // (2) logits: warp w takes k-steps [w * KS / 16, (w + 1) * KS / 16) of KS = H / 16
    {
        const int KS = P.H >> 4;
        const int k0 = warp * KS / kRouterWarps, k1 = (warp + 1) * KS / kRouterWarps;
        constexpr int NTL = NE / 8;  // 8-wide expert tiles
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const uint32_t ua = smem_u32(u_s) + (uint32_t)((lane & 15) * rb + (lane >> 4) * 16);
        const uint32_t wa = smem_u32(w_s) + (uint32_t)((lane & 7) * rb + ((lane >> 3) & 1) * 16);
        for (int kk = k0; kk < k1; ++kk) {
            uint32_t a[4], b0, b1;
            ldsm_x4_r(ua + kk * 32, a);
            ldsm_x2_r(wa + kk * 32, b0, b1);  // experts e0 .. e0+7
            mma_bf16_16816(acc[0], a, b0, b1);
            if constexpr (NTL == 2) {
                uint32_t b2, b3;
                ldsm_x2_r(wa + (uint32_t)(8 * rb) + kk * 32, b2, b3);  // experts e0+8 .. e0+15
                mma_bf16_16816(acc[1], a, b2, b3);
            }
        }
        // partial tiles: rows (tokens) lane/4 and lane/4 + 8, columns (experts) 2(lane%4), +1
        float* rw = red + warp * (16 * kRouterExp);
        const int rr = lane >> 2, cc = 2 * (lane & 3);
#pragma unroll
        for (int nt = 0; nt < NTL; ++nt) {
            rw[rr * kRouterExp + nt * 8 + cc] = acc[nt][0];
            rw[rr * kRouterExp + nt * 8 + cc + 1] = acc[nt][1];
            rw[(rr + 8) * kRouterExp + nt * 8 + cc] = acc[nt][2];
            rw[(rr + 8) * kRouterExp + nt * 8 + cc + 1] = acc[nt][3];
        }
    }
    __syncthreads();
    if (threadIdx.x < 16 * kRouterExp) {
        const int r = threadIdx.x / kRouterExp, c = threadIdx.x % kRouterExp, e = e0 + c;
        if (r < ntok && e < P.E) {
            float z = 0.f;
#pragma unroll
            for (int w = 0; w < kRouterWarps; ++w) z += red[w * (16 * kRouterExp) + r * kRouterExp + c];
            P.logits[(size_t)(tg * kRouterTok + r) * P.E + e] = z + (P.bias ? P.bias[e] : 0.f);
        }
    }

    // (3) the last CTA of the token group: top-k + softmax over the selection
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // release the CTA's logits (ordered before by the barrier)
        const uint32_t prev = atomicAdd(&P.cnt[tg], 1u);
        sh_last = (prev == gridDim.y - 1) ? 1 : 0;
        if (sh_last) {
            P.cnt[tg] = 0;
            __threadfence();  // acquire the other CTAs' logits for the whole CTA (barrier below)
        }
    }
    __syncthreads();
    if (sh_last && warp < ntok) {
        const int tl = tg * kRouterTok + warp;
        const float* z = P.logits + (size_t)tl * P.E;
        float* zs = reinterpret_cast<float*>(smem_raw) + (size_t)warp * P.E;  // u is done
        for (int ee = lane; ee < P.E; ee += 32) {
            const float v = __ldcg(z + ee);
            zs[ee] = isnan(v) ? -INFINITY : v;
        }
        __syncwarp();
        const int per = (P.E + 31) / 32;
        uint32_t taken = 0;  // bit i: candidate i * 32 + lane was selected
        float selz[8];
        int seli[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            selz[j] = -INFINITY;
            seli[j] = 0;
            if (j < P.k) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
                for (int i = 0; i < per; ++i) {
                    const int ee = i * 32 + lane;
                    if (ee < P.E && !(taken & (1u << i))) {
                        const float v = zs[ee];
                        if (v > bv || (v == bv && ee < bi)) {
                            bv = v;
                            bi = ee;
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    if (ov > bv || (ov == bv && oi < bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
                selz[j] = bv;
                seli[j] = bi;
            }
        }
        // lane j < k writes pick j: w_j = exp(z_j - z_0) / sum_i exp(z_i - z_0)
        float den = 0.f, mine = 0.f;
        int idx = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < P.k) {
                const float ex = expf(selz[j] - selz[0]);
                den += ex;
                if (lane == j) {
                    mine = ex;
                    idx = seli[j];
                }
            }
        }
        if (lane < P.k) {
            const float wj = mine / den;
            const int row_g = P.row0 + tl;
            P.idx[tl * P.k + lane] = idx;
            P.wts[tl * P.k + lane] = wj;
            if (P.user_idx) P.user_idx[(size_t)row_g * P.k + lane] = idx;
            if (P.user_w) P.user_w[(size_t)row_g * P.k + lane] = wj;
        }
    }
    task_end(ctx);
}

// ---------------------------------------------------------------------------------------
// Dispatch.  Every CTA redundantly computes the stable counting sort of the pairs
// i = t*k + j by slot (order within a slot = pair order), then gathers its share of the rows
// of u into the slot-sorted activation matrix (few rows per CTA and many loads in flight:
// the gather is latency-bound; at most kDispCtas CTAs, as each one repeats the sort).  CTA 0
// also publishes the slot offsets and pair rows.
// ---------------------------------------------------------------------------------------
constexpr int kDispRowsMin = 2;
constexpr int kDispCtas = 256;

__global__ void __launch_bounds__(256) dispatch_kernel(const DispatchProblem P, const KCtx ctx) {
    griddep_launch();
    griddep_wait();
    task_begin(ctx);
    extern __shared__ int sm_i[];
    const int R = P.nrows * P.k;
    int* pslot = sm_i;          // [R]
    int* rank = pslot + R;      // [R]
    int* row_pair = rank + R;   // [R]
    int* offs = row_pair + R;   // [E_local + 1]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < R; i += 256) {
        int gidx = P.idx[i];
        if (gidx < 0 || gidx >= P.E) {
            report(ctx, ST_BOUNDS, (uint32_t)gidx);
            gidx = 0;
        }
        pslot[i] = P.slot_map == 0 ? gidx % P.E_local : (int)(((long)gidx * P.E_local) / P.E);
    }
    __syncthreads();
    for (int s = warp; s < P.E_local; s += 8) {
        int running = 0;
        for (int c = 0; c < R; c += 32) {
            const int i = c + lane;
            const bool is = i < R && pslot[i] == s;
            const uint32_t m = __ballot_sync(0xffffffffu, is);
            if (is) rank[i] = running + __popc(m & ((1u << lane) - 1u));
            running += __popc(m);
        }
        if (lane == 0) offs[s + 1] = running;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        offs[0] = 0;
        for (int s = 0; s < P.E_local; ++s) offs[s + 1] += offs[s];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < R; i += 256) {
        const int pos = offs[pslot[i]] + rank[i];
        row_pair[pos] = i;
        if (blockIdx.x == 0) P.pair_pos[i] = pos;
    }
    if (blockIdx.x == 0)
        for (int s = threadIdx.x; s <= P.E_local; s += 256) P.offsets[s] = offs[s];
    __syncthreads();
    const int nv = P.H >> 3;
    const int rpc = (R + gridDim.x - 1) / gridDim.x;  // rows of this CTA's share
    const int rbeg = blockIdx.x * rpc;
    const int total = max(0, min(R, rbeg + rpc) - rbeg) * nv;
    constexpr int kU = 8;  // loads in flight per thread
    for (int i0 = threadIdx.x; i0 < total; i0 += 256 * kU) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = i0 + u * 256;
            if (i < total) {
                const int r = rbeg + i / nv, c = i % nv;
                const int t = row_pair[r] / P.k;
                v[u] = reinterpret_cast<const uint4*>(P.u + (size_t)(P.row0 + t) * P.H)[c];
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = i0 + u * 256;
            if (i < total) {
                const int r = rbeg + i / nv, c = i % nv;
                reinterpret_cast<uint4*>(P.xperm + (size_t)r * P.H)[c] = v[u];
            }
        }
    }
    task_end(ctx);
}

// ---------------------------------------------------------------------------------------
// Combine: out[t] = bf16(h[t] + sum_j w[t][j] * Y[pair_pos[t k + j]]), j in pick order.
// With a K-split expert-down projection, Y[r] is the sum of its K segments, formed here in
// segment order (the same fp32 operations the finishing pass would do), so that pass is not
// launched.
// ---------------------------------------------------------------------------------------
constexpr int kCombThreads = 512;
// KP: picks per token, at most.  WIDE: every pick's segment loads in flight together (few
// tokens, latency-bound); otherwise one pick at a time in fewer registers, so that two CTAs
// share an SM (many tokens).  Both perform the same fp32 operations in the same order.
template <int KP, bool WIDE>
__global__ void __launch_bounds__(kCombThreads, WIDE ? 1 : 2)
    combine_kernel(const CombineProblem P, const KCtx ctx) {
    griddep_launch();
    griddep_wait();
    task_begin(ctx);
    constexpr int kKeep = 2;  // 4-element vectors per thread kept for the fused RMSNorm (H <= 4096)
    __shared__ float red[kCombThreads / 32];
    const int tl = blockIdx.x;
    const int row = P.row0 + tl;
    const int n4 = P.H >> 2;
    int pos[KP];
    float w[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
        pos[j] = 0;
        w[j] = 0.f;
        if (j < P.k) {
            pos[j] = P.pair_pos[tl * P.k + j];
            w[j] = P.wts[tl * P.k + j];
            if (pos[j] < 0 || pos[j] >= P.nrows * P.k) {
                if (threadIdx.x == 0) report(ctx, ST_BOUNDS, (uint32_t)pos[j]);
                pos[j] = 0;
                w[j] = 0.f;
            }
        }
    }
    const uint2* h = reinterpret_cast<const uint2*>(P.h + (size_t)row * P.H);
    uint2* out = reinterpret_cast<uint2*>(P.out + (size_t)row * P.H);
    uint2 keep[kKeep];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kKeep; ++i) keep[i] = make_uint2(0, 0);
    int i = 0;
    for (int v = threadIdx.x; v < n4; v += kCombThreads, ++i) {
        // y_j = sum of pick j's K segments in segment order, then acc += w_j y_j in pick order
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const size_t sstride = (size_t)P.R * 128;
        // K segments s of a row live at ((tile * ksplit + s) * R + row) * 128 + col
        const float* base = P.Y + (size_t)((4 * v) >> 7) * P.ksplit * sstride + ((4 * v) & 127);
        if constexpr (WIDE) {
            float4 y[KP];
#pragma unroll
            for (int j = 0; j < KP; ++j) y[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (P.ksplit <= 1) {
#pragma unroll
                for (int j = 0; j < KP; ++j)
                    if (j < P.k) y[j] = *reinterpret_cast<const float4*>(P.Y + (size_t)pos[j] * P.H + 4 * v);
            } else {
                for (int s0 = 0; s0 < P.ksplit; s0 += 2) {
                    float4 ld[KP][2];
#pragma unroll
                    for (int j = 0; j < KP; ++j)
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            if (j < P.k && s0 + u < P.ksplit)
                                ld[j][u] = __ldcg(reinterpret_cast<const float4*>(
                                    base + (size_t)(s0 + u) * sstride + (size_t)pos[j] * 128));
#pragma unroll
                    for (int j = 0; j < KP; ++j)
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            if (j < P.k && s0 + u < P.ksplit) {
                                y[j].x += ld[j][u].x;
                                y[j].y += ld[j][u].y;
                                y[j].z += ld[j][u].z;
                                y[j].w += ld[j][u].w;
                            }
                }
            }
#pragma unroll
            for (int j = 0; j < KP; ++j) {
                if (j < P.k) {
                    acc[0] = fmaf(w[j], y[j].x, acc[0]);
                    acc[1] = fmaf(w[j], y[j].y, acc[1]);
                    acc[2] = fmaf(w[j], y[j].z, acc[2]);
                    acc[3] = fmaf(w[j], y[j].w, acc[3]);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < KP; ++j) {
                if (j < P.k) {
                    float4 yj;
                    if (P.ksplit <= 1) {
                        yj = *reinterpret_cast<const float4*>(P.Y + (size_t)pos[j] * P.H + 4 * v);
                    } else {
                        yj = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
                        for (int sg = 0; sg < P.ksplit; ++sg) {
                            const float4 l = __ldcg(reinterpret_cast<const float4*>(
                                base + (size_t)sg * sstride + (size_t)pos[j] * 128));
                            yj.x += l.x;
                            yj.y += l.y;
                            yj.z += l.z;
                            yj.w += l.w;
                        }
                    }
                    acc[0] = fmaf(w[j], yj.x, acc[0]);
                    acc[1] = fmaf(w[j], yj.y, acc[1]);
                    acc[2] = fmaf(w[j], yj.z, acc[2]);
                    acc[3] = fmaf(w[j], yj.w, acc[3]);
                }
            }
        }
        const uint2 hv = h[v];
        const float2 h01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hv.x));
        const float2 h23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hv.y));
        uint2 o;
        o.x = pack_bf16x2(h01.x + acc[0], h01.y + acc[1]);
        o.y = pack_bf16x2(h23.x + acc[2], h23.y + acc[3]);
        out[v] = o;
        if (P.a_next != nullptr) {
            // the next layer normalises the stored (bf16) residual
            const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.x));
            const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.y));
            ss = fmaf(x01.x, x01.x, ss);
            ss = fmaf(x01.y, x01.y, ss);
            ss = fmaf(x23.x, x23.x, ss);
            ss = fmaf(x23.y, x23.y, ss);
#pragma unroll
            for (int q = 0; q < kKeep; ++q)
                if (q == i) keep[q] = o;
        }
    }
    if (P.a_next != nullptr) {
        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int wq = 0; wq < kCombThreads / 32; ++wq) tot += red[wq];
        const float inv = rsqrtf(tot / (float)P.H + P.eps);
        const uint2* g = reinterpret_cast<const uint2*>(P.g_next);
        uint2* a = reinterpret_cast<uint2*>(P.a_next + (size_t)row * P.H);
#pragma unroll
        for (int q = 0; q < kKeep; ++q) {
            const int v = threadIdx.x + q * kCombThreads;
            if (v < n4) {
                const uint2 gv = g[v];
                const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&keep[q].x));
                const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&keep[q].y));
                const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv.x));
                const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv.y));
                uint2 r;
                r.x = pack_bf16x2(x01.x * inv * g01.x, x01.y * inv * g01.y);
                r.y = pack_bf16x2(x23.x * inv * g23.x, x23.y * inv * g23.y);
                a[v] = r;
            }
        }
    }
    task_end(ctx);
}

}  // namespace

// ---------------------------------------------------------------------------------------
// Router without device allocation (see sgp_router_topk_noalloc in sgp.h).  The scratch the
// router needs -- fp32 logits and per-token-group arrival counters -- lives in this fixed
// array; every GPU that loads the library holds it until the process exits.
// ---------------------------------------------------------------------------------------
constexpr size_t kNoallocLogits = 256 * 1024;                    // fp32 logits (1 MiB)
constexpr size_t kNoallocCounters = 256;                         // u32 token-group counters
constexpr size_t kNoallocBytes = kNoallocLogits * 4 + kNoallocCounters * 4;
static __device__ __align__(256) unsigned char g_router_scratch[kNoallocBytes];

int enqueue_rmsnorm(Launcher& L, const NormProblem& p, const KCtx& c) {
    void* args[] = {(void*)&p, (void*)&c};
    return L.launch((const void*)rmsnorm_kernel, dim3(p.nrows), dim3(256), 0, args);
}

int enqueue_router(Launcher& L, const RouterProblem& p, const KCtx& c) {
    void* args[] = {(void*)&p, (void*)&c};
    const int ne = router_experts_per_cta(p.H, p.E, p.nrows);
    dim3 grid((p.nrows + kRouterTok - 1) / kRouterTok, (p.E + ne - 1) / ne);
    return L.launch(ne == 16 ? (const void*)router_kernel<16> : (const void*)router_kernel<8>, grid,
                    dim3(kRouterWarps * 32),
                    router_smem_bytes(p.H, p.E, ne), args);
}

int enqueue_dispatch(Launcher& L, const DispatchProblem& p, const KCtx& c) {
    void* args[] = {(void*)&p, (void*)&c};
    const int R = p.nrows * p.k;
    dim3 grid(std::max(1, std::min((R + kDispRowsMin - 1) / kDispRowsMin, kDispCtas)));
    return L.launch((const void*)dispatch_kernel, grid, dim3(256),
                    (size_t)(3 * R + p.E_local + 1) * sizeof(int), args);
}

// ---------------------------------------------------------------------------------------
// Virtual communication (a collective of a multi-GPU deployment emulated on one GPU): the
// local endpoint work -- the payload is read and written to scratch -- and a duration of at
// least the model's floor, measured from the moment the payload is ready.  Every CTA copies
// its share, then sleeps until its own floor has passed (bounded by the floor itself).
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) comm_kernel(const CommProblem P, const KCtx ctx) {
    griddep_launch();
    griddep_wait();
    task_begin(ctx);
    const uint64_t t0 = globaltimer();
    const size_t n16 = P.bytes / 16;
    const uint4* __restrict__ src = reinterpret_cast<const uint4*>(P.src);
    uint4* __restrict__ dst = reinterpret_cast<uint4*>(P.dst);
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    constexpr int kU = 4;  // independent loads in flight per thread
    for (size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n16; i0 += kU * stride) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (i0 + u * stride < n16) v[u] = __ldcg(src + i0 + u * stride);
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (i0 + u * stride < n16) dst[i0 + u * stride] = v[u];
    }
    __syncthreads();
    if (threadIdx.x == 0)
        while (globaltimer() - t0 < P.floor_ns) __nanosleep(256);
    __syncthreads();
    task_end(ctx);
}

// ---------------------------------------------------------------------------------------
// L2 prefetch of the weights of a coming projection, run beside the chain while the kernels
// before that projection leave HBM idle (a finishing pass, the router and dispatch, the
// combine).  Consecutive chunks go to different CTAs, so the bulk prefetches are issued by
// the TMA units of many SMs at once.
// ---------------------------------------------------------------------------------------
constexpr uint32_t kPrefetchChunk = 32768;

__global__ void __launch_bounds__(32) prefetch_kernel(const PrefetchProblem P, const KCtx ctx) {
    griddep_launch();
    griddep_wait();
    task_begin(ctx);
    const uint64_t pol = policy_evict_last();
    const size_t n0 = (P.bytes[0] + kPrefetchChunk - 1) / kPrefetchChunk;
    const size_t n1 = (P.bytes[1] + kPrefetchChunk - 1) / kPrefetchChunk;
    for (size_t c = (size_t)threadIdx.x * gridDim.x + blockIdx.x; c < n0 + n1;
         c += (size_t)gridDim.x * blockDim.x) {
        const bool first = c < n0;
        const size_t off = (first ? c : c - n0) * kPrefetchChunk;
        const size_t left = (first ? P.bytes[0] : P.bytes[1]) - off;
        const uint32_t nb = (uint32_t)(left < kPrefetchChunk ? left : kPrefetchChunk);
        const char* src = static_cast<const char*>(first ? P.base[0] : P.base[1]) + off;
        asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src),
                     "r"(nb), "l"(pol)
                     : "memory");
    }
    task_end(ctx);
}

int enqueue_prefetch(Launcher& L, const PrefetchProblem& p, const KCtx& c) {
    for (int r = 0; r < 2; ++r)
        if ((reinterpret_cast<uintptr_t>(p.base[r]) & 15) || (p.bytes[r] & 15) ||
            (p.bytes[r] && !p.base[r]))
            return (int)cudaErrorInvalidValue;
    if (p.bytes[0] + p.bytes[1] == 0) return 0;
    void* args[] = {(void*)&p, (void*)&c};
    return L.launch_side((const void*)prefetch_kernel, dim3(std::max(1, p.grid)), dim3(32), 0,
                         args);
}

int enqueue_comm(Launcher& L, const CommProblem& p, const KCtx& c) {
    if (((reinterpret_cast<uintptr_t>(p.src) | reinterpret_cast<uintptr_t>(p.dst)) & 15) ||
        p.floor_ns > 1000000000ull)
        return (int)cudaErrorInvalidValue;
    void* args[] = {(void*)&p, (void*)&c};
    return L.launch((const void*)comm_kernel, dim3(32), dim3(256), 0, args);
}

int enqueue_combine(Launcher& L, const CombineProblem& p, const KCtx& c) {
    void* args[] = {(void*)&p, (void*)&c};
    if (p.k < 1 || p.k > 8 || (p.H & 3) || (p.a_next != nullptr && p.H > 4 * 2 * kCombThreads))
        return (int)cudaErrorInvalidValue;
    const bool wide = p.nrows <= 96;  // few tokens: load latency, not occupancy, is the limit
    const void* f = p.k <= 4 ? (wide ? (const void*)combine_kernel<4, true> : (const void*)combine_kernel<4, false>)
                             : (wide ? (const void*)combine_kernel<8, true> : (const void*)combine_kernel<8, false>);
    return L.launch(f, dim3(p.nrows), dim3(kCombThreads), 0, args);
}

}  // namespace sgp

// Host side of the allocation-free router.  Once per device (with that device current) the
// set-up looks up the device address of g_router_scratch and prepares both router kernel
// instances for the largest dynamic shared memory the device allows, so that no later call
// touches a kernel attribute; the per-instance limits decide which sizes are refused.
namespace {
struct NoallocDev {
    bool ready = false;
    void* scratch = nullptr;
    size_t smem_limit[2] = {0, 0};  // router_kernel<8>, router_kernel<16>
};
std::mutex g_noalloc_mu;
NoallocDev g_noalloc[128];

int noalloc_setup(int dev, NoallocDev& s) {
    using namespace sgp;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_router_scratch) != cudaSuccess || p == nullptr)
        return SGP_ERR_CUDA;
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return SGP_ERR_CUDA;
    const void* fns[2] = {(const void*)router_kernel<8>, (const void*)router_kernel<16>};
    for (int i = 0; i < 2; ++i) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, fns[i]) != cudaSuccess) return SGP_ERR_CUDA;
        const int dyn = optin - (int)fa.sharedSizeBytes;
        if (dyn <= 0 ||
            cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
            return SGP_ERR_CUDA;
        s.smem_limit[i] = (size_t)dyn;
    }
    s.scratch = p;
    s.ready = true;
    return SGP_OK;
}
}  // namespace

extern "C" int sgp_router_topk_noalloc(const sgp_dims* d, const void* h, const void* g_mlp,
                                       const void* w_router, const float* router_bias,
                                       int n_tokens, void* u_out, int32_t* topk_idx,
                                       float* topk_w, sgp_stream_t stream) {
    using namespace sgp;
    if (!d || !h || !g_mlp || !w_router || !u_out || !topk_idx || !topk_w)
        return SGP_ERR_INVALID_ARG;
    if (d->hidden <= 0 || d->hidden % 64 || d->hidden > 4096 || d->top_k < 1 || d->top_k > 8 ||
        d->n_experts < d->top_k || d->n_experts > 1024 || !(d->rms_eps > 0.f))
        return SGP_ERR_INVALID_ARG;
    const void* ptrs[] = {h, g_mlp, w_router, u_out};
    for (const void* q : ptrs)
        if (reinterpret_cast<uintptr_t>(q) & 15) return SGP_ERR_INVALID_ARG;
    const int groups = (n_tokens + kRouterTok - 1) / kRouterTok;
    // sizes beyond the fixed scratch are refused; nothing is launched
    if (n_tokens < 1 || (size_t)n_tokens * d->n_experts > kNoallocLogits ||
        (size_t)groups > kNoallocCounters)
        return SGP_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return SGP_ERR_CUDA;
    NoallocDev st;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc[dev].ready) {
            const int r = noalloc_setup(dev, g_noalloc[dev]);
            if (r != SGP_OK) return r;
        }
        st = g_noalloc[dev];
    }
    const int ne = router_experts_per_cta(d->hidden, d->n_experts, n_tokens);
    const size_t smem = router_smem_bytes(d->hidden, d->n_experts, ne);
    if (smem > st.smem_limit[ne == 16 ? 1 : 0]) return SGP_ERR_INVALID_ARG;  // nothing launched
    float* logits = reinterpret_cast<float*>(st.scratch);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(logits + kNoallocLogits);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the arrival counters must start at zero; the logits need no clearing
    if (cudaMemsetAsync(cnt, 0, kNoallocCounters * 4, s) != cudaSuccess) return SGP_ERR_CUDA;
    RouterProblem p;
    memset(&p, 0, sizeof(p));
    p.h = reinterpret_cast<const bf16*>(h);
    p.g = reinterpret_cast<const bf16*>(g_mlp);
    p.u = reinterpret_cast<bf16*>(u_out);
    p.Wr = reinterpret_cast<const bf16*>(w_router);
    p.bias = router_bias;
    p.logits = logits;
    p.idx = topk_idx;
    p.wts = topk_w;
    p.cnt = cnt;
    p.row0 = 0;
    p.nrows = n_tokens;
    p.H = d->hidden;
    p.E = d->n_experts;
    p.k = d->top_k;
    p.eps = d->rms_eps;
    // the router kernel has no device-side error path (no waits, no data-dependent indexing
    // beyond the sizes checked above), so it gets no status word
    KCtx c;
    memset(&c, 0, sizeof(c));
    c.timeout_ns = 2000000000ull;
    const void* fn = ne == 16 ? (const void*)router_kernel<16> : (const void*)router_kernel<8>;
    void* args[] = {(void*)&p, (void*)&c};
    dim3 grid(groups, (d->n_experts + ne - 1) / ne);
    if (cudaLaunchKernel(fn, grid, dim3(kRouterWarps * 32), args, smem, s) != cudaSuccess)
        return SGP_ERR_CUDA;
    return SGP_OK;
}
