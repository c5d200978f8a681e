// GQA decode attention over a bf16 KV cache, split along the sequence (split-KV).
//
// Persistent: gridDim.x CTAs (one per SM of the pool), each of kAWarps independent streaming
// warps.  The work is the flat list of chunks (sequence, KV head, chunk of P.chunk
// positions); warp w of the grid owns a contiguous, equal share of that list, so the split
// of work follows the pool size while every chunk's arithmetic does not.
//
// Every warp streams its chunks through a private shared-memory stage of POS positions: a K
// half and a V half, one TMA operation each (L2 evict-first), refilled by lane 0; a warp never
// waits on another.  Two refill schedules, the same arithmetic:
//   split (P.kv_split): each half has its own mbarrier; the K half takes the next stage's keys
//     as soon as the scores are computed, so that load overlaps the softmax and the V
//     product, and the V half is refilled once that product is done, overlapping the next
//     scores.  Faster alone on the GPU (both configurations) and in a partial pool with
//     128-position stages;
//   joint: one mbarrier, both halves refilled after the V product.  Gentler on the HBM a
//     neighbouring stage shares: with 64-position stages on a partial pool, the split
//     schedule made the attention faster alone but the two-stage pipeline slower.
// A warp's arithmetic on a stage takes about as long as the stage's load, so shared memory is
// spent on more warps rather than on deeper per-warp buffering: twelve warps with one
// 64-position stage each stream faster on a partial pool than six with 128 positions, six
// with 128 faster on the full GPU when each warp gets only a few chunks, and six with one
// stage faster than three with two.
// Per stage the warp computes, on warp-level bf16 MMAs with fp32 accumulation,
//     S^T = K q^T   (M = 16 positions, N = 8 query heads of the KV head, K = 64)
//     O^T += V^T P^T (M = 16 dims, N = 8 heads, K = 16 positions),
// i.e. the G query heads that share a KV head are the MMA's N dimension, so no tensor work
// is spent on padding rows.  P goes from the accumulator layout of S^T to the operand layout
// of the second product with movmatrix (an in-register 8x8 transpose).  An online softmax
// (max over positions per head, base 2) runs between the two products.
//
// A chunk ends with its partial (running max, sum, unnormalised O) written to the workspace;
// the warp that completes the last chunk of a (sequence, KV head) merges all its chunks in
// chunk order (log-sum-exp combine).  Chunking and merge order are fixed by the shape, so the
// output does not depend on the grid or on scheduling.  The same merge is the
// partial-attention aggregation used when a sequence is split across partitions
// ("Starscream: Reimagining LLM Sharding on AMD Instinct GPUs with GPU Partitioning",
// sequence-length-sharded attention).
#include "kernels.h"

namespace sgp {

namespace {

// Two configurations of the same kernel, chosen per shape (never per pool: the stage
// length sets the order of the fp32 online softmax): NW streaming warps per CTA with one
// stage of POS positions each, 192 KB of ring either way.
//   12 x 64: twice the warps on half the arithmetic per stage -- faster per SM where the pool
//            is small and there are many chunks (long caches);
//    6 x 128: larger TMA boxes -- faster on the full GPU when chunks per warp are few.
constexpr int kAMaxRows = 512;               // sequences per launch (prefix table size)
constexpr int kAPerLane = kAMaxRows / 32;    // sequences per lane of the prefix scan

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk `ch` of row `r` in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
    return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
}

// Where a warp stands in its share of the chunk list.
struct Cursor {
    int i;               // chunk index (>= end: done)
    int t, kvh, c, S_t;  // sequence (launch-local), KV head, chunk of that pair, chunks/pair
    int p0, p1;          // positions [p0, p1) of the chunk
    int j, nst;          // stage within the chunk, stages of the chunk
};

template <int POS>
__device__ __forceinline__ void cursor_at(Cursor& x, int i, const int* pre, const int* kvl,
                                          int nrows, const AttnProblem& P) {
    x.i = i;
    int lo = 0, hi = nrows;  // largest t with pre[t] <= i  (pre[nrows] = total > i)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= i) lo = mid;
        else hi = mid;
    }
    x.t = lo;
    x.S_t = (pre[lo + 1] - pre[lo]) / P.nkv;
    const int r = i - pre[lo];
    x.kvh = r / x.S_t;
    x.c = r - x.kvh * x.S_t;
    const int L = kvl[lo];
    const int first = P.window > 0 ? max(0, L - P.window) : 0;
    x.p0 = first + x.c * P.chunk;
    x.p1 = min(L, x.p0 + P.chunk);
    x.j = 0;
    x.nst = (x.p1 - x.p0 + POS - 1) / POS;
}

template <int NT>
__device__ void merge_pair(const AttnProblem& P, int t, int kvh, int S_t, int lane) {
    // lane -> head hl (fixed), dims d = lane / Gp + k * (32 / Gp)
    constexpr int Gp = NT * 8;
    constexpr int kPer = 64 * Gp / 32;
    const int hl = lane % Gp, d0 = lane / Gp;
    const size_t pair = (size_t)t * P.nkv + kvh;
    const float* bml = P.part_ml + pair * P.S_max * 32;
    const float* bacc = P.part_acc + pair * P.S_max * 64 * 16;
    float M = -INFINITY;
    for (int c = 0; c < S_t; ++c) M = fmaxf(M, __ldcg(bml + c * 32 + 2 * hl));
    float O[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) O[k] = 0.f;
    float Ls = 0.f;
    int c = 0;
    for (; c + 2 <= S_t; c += 2) {
        const float m0 = __ldcg(bml + c * 32 + 2 * hl), l0 = __ldcg(bml + c * 32 + 2 * hl + 1);
        const float m1 = __ldcg(bml + (c + 1) * 32 + 2 * hl);
        const float l1 = __ldcg(bml + (c + 1) * 32 + 2 * hl + 1);
        float a0[kPer], a1[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int d = d0 + k * (32 / Gp);
            a0[k] = __ldcg(bacc + ((size_t)c * 64 + d) * 16 + hl);
            a1[k] = __ldcg(bacc + ((size_t)(c + 1) * 64 + d) * 16 + hl);
        }
        const float w0 = exp2f(m0 - M), w1 = exp2f(m1 - M);
        Ls = fmaf(w0, l0, Ls);
        Ls = fmaf(w1, l1, Ls);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            O[k] = fmaf(w0, a0[k], O[k]);
            O[k] = fmaf(w1, a1[k], O[k]);
        }
    }
    for (; c < S_t; ++c) {
        const float m0 = __ldcg(bml + c * 32 + 2 * hl), l0 = __ldcg(bml + c * 32 + 2 * hl + 1);
        const float w0 = exp2f(m0 - M);
        Ls = fmaf(w0, l0, Ls);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int d = d0 + k * (32 / Gp);
            O[k] = fmaf(w0, __ldcg(bacc + ((size_t)c * 64 + d) * 16 + hl), O[k]);
        }
    }
    if (hl < P.G) {
        const float inv = 1.f / Ls;
        bf16* o = P.o + (size_t)(P.row0 + t) * (P.nq * 64) + (size_t)(kvh * P.G + hl) * 64;
#pragma unroll
        for (int k = 0; k < kPer; ++k) o[d0 + k * (32 / Gp)] = __float2bfloat16_rn(O[k] * inv);
    }
}

template <int NT, int NW, int POS, bool SPLIT>
__global__ void __launch_bounds__(NW * 32, 1)
    attn_decode_kernel(const __grid_constant__ AttnProblem P, const KCtx ctx) {
    constexpr int kAWarps = NW;                    // streaming warps per CTA
    constexpr int kAPos = POS;                     // positions per stage
    constexpr int kAPT = kAPos / 16;               // 16-position MMA tiles per stage
    constexpr int kAHalf = kAPos * 128;            // K (or V) bytes of a stage
    constexpr int kAStage = 2 * kAHalf;            // K then V
    constexpr size_t kARing = (size_t)kAWarps * kAStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kARing);  // [warp][K, V]
    int* pre = reinterpret_cast<int*>(full + kAWarps * 2);        // [kAMaxRows + 1]
    int* kvl = pre + kAMaxRows + 1;                                 // [kAMaxRows]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    griddep_launch();

    // ---- chunk counts and their prefix over the launch's sequences (warp 0) ----
    // kv_len is an input of the call, never written by a kernel: this prologue may run while
    // the previous kernel (the QKV projection's last launch) still runs.
    if (warp == 0) {
        int cnt[kAPerLane], sum = 0;
#pragma unroll
        for (int k = 0; k < kAPerLane; ++k) {
            const int t = lane * kAPerLane + k;
            cnt[k] = 0;
            if (t < P.nrows) {
                const int L = P.kv_len[P.row0 + t];
                kvl[t] = L;
                if (L < 1 || L > P.cap) {
                    if (blockIdx.x == 0) report(ctx, ST_BOUNDS, (uint32_t)L);
                } else {
                    const int first = P.window > 0 ? max(0, L - P.window) : 0;
                    const int S = (L - first + P.chunk - 1) / P.chunk;
                    if (S > P.S_max) {
                        if (blockIdx.x == 0) report(ctx, ST_BOUNDS, (uint32_t)S);
                    } else {
                        cnt[k] = S * P.nkv;
                    }
                }
            }
            sum += cnt[k];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
#pragma unroll
        for (int k = 0; k < kAPerLane; ++k) {
            const int t = lane * kAPerLane + k;
            if (t < P.nrows) pre[t] = run;
            run += cnt[k];
        }
        if (lane == 31) pre[P.nrows] = incl;
        if (lane < 2 * kAWarps) mbar_init(&full[lane], 1);
        fence_barrier_init();
        if (lane == 0) {
            prefetch_tensormap(&P.tmK);
            prefetch_tensormap(&P.tmV);
        }
    }
    __syncthreads();
    // q and the appended KV row come from the previous kernel
    griddep_wait();
    task_begin(ctx);

    const int total = pre[P.nrows];
    const long long W = (long long)gridDim.x * kAWarps;
    const long long gw = (long long)blockIdx.x * kAWarps + warp;
    const int i0 = (int)(gw * total / W), i1 = (int)((gw + 1) * total / W);

    uint8_t* ring = smem + (size_t)warp * kAStage;
    uint64_t* barK = full + warp * 2;
    uint64_t* barV = barK + 1;
    const uint64_t pol = policy_evict_first();
    const int g = lane >> 2, cq = lane & 3;

    Cursor cs, ld;
    if (i0 < i1) cursor_at<POS>(cs, i0, pre, kvl, P.nrows, P);
    else cs.i = i1;
    ld = cs;
    // K and V halves of stage n arrive on barK / barV phase n & 1; `ld` is the next stage
    // whose K half is to be issued, v_row the cache row of the stage whose V half is pending
    // (joint schedule: both halves on barK, issued together by issue_k)
    uint32_t n_k = 0, n_v = 0;  // K / V halves issued (n_v stays 0 when joint)
    uint32_t n_kc = 0, n_con = 0;  // K halves consumed, stages consumed
    int v_row = 0;
    auto issue_k = [&]() {  // K half (joint: the whole stage) of stage `ld`, then advance `ld`
        const int row = ((P.row0 + ld.t) * P.nkv + ld.kvh) * P.cap + ld.p0 + ld.j * kAPos;
        if (lane == 0) {
            mbar_arrive_expect_tx(barK, SPLIT ? kAHalf : kAStage);
            tma_load_2d(ring, &P.tmK, barK, 0, row, pol);
            if constexpr (!SPLIT) tma_load_2d(ring + kAHalf, &P.tmV, barK, 0, row, pol);
        }
        v_row = row;
        ++n_k;
        if (++ld.j == ld.nst) {
            if (ld.i + 1 < i1) cursor_at<POS>(ld, ld.i + 1, pre, kvl, P.nrows, P);
            else ld.i = i1;
        }
    };
    auto issue_v = [&]() {  // V half of the stage whose K half was issued last
        if (lane == 0) {
            mbar_arrive_expect_tx(barV, kAHalf);
            tma_load_2d(ring + kAHalf, &P.tmV, barV, 0, v_row, pol);
        }
        ++n_v;
    };
    if (ld.i < i1) {
        issue_k();
        if constexpr (SPLIT) issue_v();
    }

    uint32_t qf[NT][4][2];
    int q_t = -1, q_h = -1;
    float m_run[NT][2], l_run[NT][2], oacc[4][NT][4];
    bool failed = false;

    while (cs.i < i1) {
        if (cs.j == 0) {
            if (cs.t != q_t || cs.kvh != q_h) {  // query fragments of the new (sequence, KV head)
                q_t = cs.t;
                q_h = cs.kvh;
                const bf16* qa =
                    P.q + (size_t)(P.row0 + cs.t) * (P.nq * 64) + (size_t)(cs.kvh * P.G) * 64;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int h = nt * 8 + g;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int col = kk * 16 + 2 * cq;
                        qf[nt][kk][0] = h < P.G ? *reinterpret_cast<const uint32_t*>(qa + h * 64 + col) : 0u;
                        qf[nt][kk][1] =
                            h < P.G ? *reinterpret_cast<const uint32_t*>(qa + h * 64 + col + 8) : 0u;
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                m_run[nt][0] = m_run[nt][1] = -INFINITY;
                l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
                for (int md = 0; md < 4; ++md)
                    oacc[md][nt][0] = oacc[md][nt][1] = oacc[md][nt][2] = oacc[md][nt][3] = 0.f;
            }
        }
        const bool okk = mbar_wait(barK, n_con & 1u, ctx.timeout_ns);
        if (__any_sync(0xffffffffu, !okk)) {
            if (lane == 0) report(ctx, ST_TIMEOUT, 10);
            failed = true;
            break;
        }
        if constexpr (SPLIT) ++n_kc;
        const uint32_t ka = smem_u32(ring), va = ka + kAHalf;
        const int valid = min(kAPos, cs.p1 - (cs.p0 + cs.j * kAPos));
        // positions past the chunk: zero V (the cache there is arbitrary, P is 0 there);
        // joint: V has landed with K
        auto zero_v_tail = [&]() {
            if (valid < kAPos) {
                uint4* v4 = reinterpret_cast<uint4*>(ring + kAHalf);
                for (int e = valid * 8 + lane; e < kAPos * 8; e += 32) v4[e] = make_uint4(0, 0, 0, 0);
                __syncwarp();
            }
        };
        if constexpr (!SPLIT) zero_v_tail();

        // ---- S^T = K q^T: 8 position tiles x NT head tiles ----
        float s[kAPT][NT][4];
#pragma unroll
        for (int mt = 0; mt < kAPT; ++mt) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) s[mt][nt][0] = s[mt][nt][1] = s[mt][nt][2] = s[mt][nt][3] = 0.f;
            const int r = mt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t a[4];
                ldsm_x4(ka + sw128(r, kk * 2 + (lane >> 4)), a);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816(s[mt][nt], a, qf[nt][kk][0], qf[nt][kk][1]);
            }
        }
        // ---- online softmax over this stage's positions (heads 2cq, 2cq+1 of each tile) ----
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < kAPT; ++mt) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float v0 = s[mt][nt][2 * hf] * P.scale_log2;
                    float v1 = s[mt][nt][2 * hf + 1] * P.scale_log2;
                    if (valid < kAPos && mt * 16 + hf * 8 + g >= valid) v0 = v1 = -INFINITY;
                    s[mt][nt][2 * hf] = v0;
                    s[mt][nt][2 * hf + 1] = v1;
                    mx0 = fmaxf(mx0, v0);
                    mx1 = fmaxf(mx1, v1);
                }
            }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float n0 = fmaxf(m_run[nt][0], mx0), n1 = fmaxf(m_run[nt][1], mx1);
            const float c0 = m_run[nt][0] == -INFINITY ? 0.f : exp2f(m_run[nt][0] - n0);
            const float c1 = m_run[nt][1] == -INFINITY ? 0.f : exp2f(m_run[nt][1] - n1);
            m_run[nt][0] = n0;
            m_run[nt][1] = n1;
            float r0 = 0.f, r1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < kAPT; ++mt) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float e0 = exp2f(s[mt][nt][2 * hf] - n0);
                    const float e1 = exp2f(s[mt][nt][2 * hf + 1] - n1);
                    s[mt][nt][2 * hf] = e0;
                    s[mt][nt][2 * hf + 1] = e1;
                    r0 += e0;
                    r1 += e1;
                }
            }
            // per-lane partial sums; reduced over the position lanes at the end of the chunk
            l_run[nt][0] = l_run[nt][0] * c0 + r0;
            l_run[nt][1] = l_run[nt][1] * c1 + r1;
#pragma unroll
            for (int md = 0; md < 4; ++md) {
                oacc[md][nt][0] *= c0;
                oacc[md][nt][1] *= c1;
                oacc[md][nt][2] *= c0;
                oacc[md][nt][3] *= c1;
            }
        }
        if constexpr (SPLIT) {
            // ---- K half consumed: the next stage's keys load during the V product ----
            fence_proxy_async();
            __syncwarp();
            if (ld.i < i1) issue_k();
            const bool okv = mbar_wait(barV, n_con & 1u, ctx.timeout_ns);
            if (__any_sync(0xffffffffu, !okv)) {
                if (lane == 0) report(ctx, ST_TIMEOUT, 11);
                failed = true;
                break;
            }
            zero_v_tail();
        }
        // ---- O^T += V^T P^T: 8 position steps of 16 x 4 dim tiles x NT head tiles ----
#pragma unroll
        for (int ks = 0; ks < kAPT; ++ks) {
            uint32_t b0[NT], b1[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                b0[nt] = movmatrix_t(pack_bf16x2(s[ks][nt][0], s[ks][nt][1]));
                b1[nt] = movmatrix_t(pack_bf16x2(s[ks][nt][2], s[ks][nt][3]));
            }
            const int r = ks * 16 + ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
            for (int md = 0; md < 4; ++md) {
                uint32_t a[4];
                ldsm_x4_t(va + sw128(r, md * 2 + ((lane >> 3) & 1)), a);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816(oacc[md][nt], a, b0[nt], b1[nt]);
            }
        }
        // ---- V half consumed (split: the next stage's values load during its scores;
        //      joint: the whole stage is refilled) ----
        fence_proxy_async();
        __syncwarp();
        ++n_con;
        if constexpr (SPLIT) {
            if (n_v < n_k) issue_v();
        } else if (ld.i < i1) {
            issue_k();
        }

        if (cs.j == cs.nst - 1) {
            // ---- end of chunk: row sums over the position lanes, then partial or output ----
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    l_run[nt][0] += __shfl_xor_sync(0xffffffffu, l_run[nt][0], o);
                    l_run[nt][1] += __shfl_xor_sync(0xffffffffu, l_run[nt][1], o);
                }
            const size_t pair = (size_t)cs.t * P.nkv + cs.kvh;
            if (cs.S_t == 1) {
                bf16* o = P.o + (size_t)(P.row0 + cs.t) * (P.nq * 64) + (size_t)(cs.kvh * P.G) * 64;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int h = nt * 8 + 2 * cq;
                    const float i0f = 1.f / l_run[nt][0], i1f = 1.f / l_run[nt][1];
#pragma unroll
                    for (int md = 0; md < 4; ++md) {
                        const int d = md * 16 + g;
                        if (h < P.G) {
                            o[h * 64 + d] = __float2bfloat16_rn(oacc[md][nt][0] * i0f);
                            o[h * 64 + d + 8] = __float2bfloat16_rn(oacc[md][nt][2] * i0f);
                        }
                        if (h + 1 < P.G) {
                            o[(h + 1) * 64 + d] = __float2bfloat16_rn(oacc[md][nt][1] * i1f);
                            o[(h + 1) * 64 + d + 8] = __float2bfloat16_rn(oacc[md][nt][3] * i1f);
                        }
                    }
                }
            } else {
                float* pml = P.part_ml + (pair * P.S_max + cs.c) * 32;
                float* pacc = P.part_acc + (pair * P.S_max + cs.c) * 64 * 16;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int h = nt * 8 + 2 * cq;
#pragma unroll
                    for (int md = 0; md < 4; ++md) {
                        const int d = md * 16 + g;
                        *reinterpret_cast<float2*>(pacc + d * 16 + h) =
                            make_float2(oacc[md][nt][0], oacc[md][nt][1]);
                        *reinterpret_cast<float2*>(pacc + (d + 8) * 16 + h) =
                            make_float2(oacc[md][nt][2], oacc[md][nt][3]);
                    }
                    if (g == 0)
                        *reinterpret_cast<float4*>(pml + 2 * h) =
                            make_float4(m_run[nt][0], l_run[nt][0], m_run[nt][1], l_run[nt][1]);
                }
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    const uint32_t prev = atomicAdd(&P.cnt[pair], 1u);
                    last = prev == (uint32_t)cs.S_t - 1;
                    if (last) P.cnt[pair] = 0;
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence();
                    merge_pair<NT>(P, cs.t, cs.kvh, cs.S_t, lane);
                }
            }
        }
        if (++cs.j == cs.nst) {
            if (cs.i + 1 < i1) cursor_at<POS>(cs, cs.i + 1, pre, kvl, P.nrows, P);
            else cs.i = i1;
        }
    }
    if (failed) {
        // drain this warp's loads still in flight (bounded): at most one per half, the
        // stage the warp was waiting on or the one after it
        for (uint32_t q = SPLIT ? n_kc : n_con; q < n_k; ++q)
            (void)mbar_wait(barK, q & 1u, 10000000ull);
        for (uint32_t q = n_con; q < n_v; ++q) (void)mbar_wait(barV, q & 1u, 10000000ull);
    }
    task_end(ctx);
}

}  // namespace

int enqueue_attention(Launcher& L, const AttnProblem& p, const KCtx& c) {
    if (p.nrows < 1 || p.nrows > kAMaxRows || p.G < 1 || p.G > 16 ||
        (p.pos != 64 && p.pos != 128) || p.chunk % p.pos)
        return (int)cudaErrorInvalidValue;
    const int nw = p.pos == 64 ? 12 : 6;
    dim3 grid(p.n_cta > 0 ? p.n_cta : 1), block(nw * 32);
    const size_t smem = (size_t)nw * 2 * p.pos * 128 + 1024 + nw * 2 * 8 +
                        (2 * kAMaxRows + 1) * 4;
    void* args[] = {(void*)&p, (void*)&c};
    // [pos == 64][G > 8][kv_split]
    static const void* const kern[2][2][2] = {
        {{(const void*)attn_decode_kernel<1, 6, 128, false>, (const void*)attn_decode_kernel<1, 6, 128, true>},
         {(const void*)attn_decode_kernel<2, 6, 128, false>, (const void*)attn_decode_kernel<2, 6, 128, true>}},
        {{(const void*)attn_decode_kernel<1, 12, 64, false>, (const void*)attn_decode_kernel<1, 12, 64, true>},
         {(const void*)attn_decode_kernel<2, 12, 64, false>, (const void*)attn_decode_kernel<2, 12, 64, true>}}};
    const void* f = kern[p.pos == 64][p.G > 8][p.kv_split != 0];
    return L.launch(f, grid, block, smem, args, true);
}

}  // namespace sgp
