// GQA decode attention over a bf16 KV cache, split along the sequence (split-KV).
//
// One CTA = (sequence, KV head, chunk of kAttnChunk positions).  The KV cache is pure
// streaming traffic, so it goes HBM -> shared memory by TMA with an L2 evict-first hint, in
// stages of 128 positions: one 16 KB TMA operation for K and one for V (the per-SM rate of
// TMA grows with the size of each operation), two stages in flight per CTA.  The four warps
// split each stage (32 positions each) and release it through an "empty" barrier; one thread
// refills it.  The G query heads that share a KV head form the M = 16 rows of warp-level
// bf16 MMAs (rows >= G are zero): S = q K^T and O += P V with fp32 accumulation, an online
// softmax with quad-shuffle row reductions in between.  The warps merge in a fixed order; a
// sequence's chunks are merged (log-sum-exp combine) in chunk order by the last CTA to
// finish, so the result does not depend on scheduling.  The same merge is the
// partial-attention aggregation used when a sequence is split across partitions
// ("Starscream: Reimagining LLM Sharding on AMD Instinct GPUs with GPU Partitioning",
// sequence-length-sharded attention).
#include "kernels.h"

namespace sgp {

namespace {

constexpr int kWarps = 4;
constexpr int kStagePos = 128;                // positions per stage
constexpr int kHalfBytes = kStagePos * 128;   // K (or V) of one stage: 16 KB
constexpr int kStageBytes = 2 * kHalfBytes;   // K then V
constexpr int kStages = 2;
constexpr int kSub = kStagePos / kWarps;      // positions per warp per stage

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
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

__global__ void __launch_bounds__(kWarps * 32)
    attn_decode_kernel(const __grid_constant__ AttnProblem P, const KCtx ctx) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    int* sh_last = reinterpret_cast<int*>(empty + kStages);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x, kvh = blockIdx.y, tl = blockIdx.z;
    const int t = P.row0 + tl;
    task_begin(ctx);

    const int L = P.kv_len[t];
    if (L < 1 || L > P.cap) {
        if (tid == 0) report(ctx, ST_BOUNDS, (uint32_t)L);
        task_end(ctx);
        return;
    }
    const int lo = P.window > 0 ? max(0, L - P.window) : 0;
    const int S_t = (L - lo + P.chunk - 1) / P.chunk;
    if (s >= S_t || S_t > P.S_max) {
        if (S_t > P.S_max && tid == 0 && s == 0) report(ctx, ST_BOUNDS, (uint32_t)S_t);
        task_end(ctx);
        return;
    }
    const int p0 = lo + s * P.chunk;
    const int p1 = min(L, p0 + P.chunk);
    const int nstage = (p1 - p0 + kStagePos - 1) / kStagePos;
    const int row_base = (t * P.nkv + kvh) * P.cap + p0;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        fence_barrier_init();
        prefetch_tensormap(&P.tmK);
        prefetch_tensormap(&P.tmV);
    }
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    auto issue = [&](int i) {  // stage i -> ring slot i % kStages
        uint8_t* sk = smem + (i % kStages) * kStageBytes;
        uint64_t* bar = &full[i % kStages];
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d(sk, &P.tmK, bar, 0, row_base + i * kStagePos, pol);
        tma_load_2d(sk + kHalfBytes, &P.tmV, bar, 0, row_base + i * kStagePos, pol);
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < kStages && issued < nstage; ++issued) issue(issued);

    // query fragments (A operand, 16 rows x 64): rows g < G are the heads of this KV head
    const int G = P.G;
    const bool rows_b = G > 8;  // rows 8..15 hold heads only when a group exceeds 8
    const int hA = lane >> 2, hB = hA + 8;
    uint32_t aq[4][4];
    {
        const bf16* qa = P.q + (size_t)t * (P.nq * 64) + (size_t)(kvh * G) * 64;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int c = kk * 16 + 2 * (lane & 3);
            auto ld2 = [&](int h, int col) -> uint32_t {
                if (h >= G) return 0u;
                return *reinterpret_cast<const uint32_t*>(qa + (size_t)h * 64 + col);
            };
            aq[kk][0] = ld2(hA, c);
            aq[kk][1] = ld2(hB, c);
            aq[kk][2] = ld2(hA, c + 8);
            aq[kk][3] = ld2(hB, c + 8);
        }
    }

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float oacc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    bool failed = false;

    for (int i = 0; i < nstage; ++i) {
        const int st = i % kStages;
        const uint32_t par = (uint32_t)(i / kStages) & 1u;
        if (!mbar_wait(&full[st], par, ctx.timeout_ns)) {
            if (lane == 0) report(ctx, ST_TIMEOUT, 10);
            failed = true;
        }
        failed = __any_sync(0xffffffffu, failed);
        if (failed) break;
        // this warp's 32 positions of the stage
        uint8_t* sk = smem + st * kStageBytes + warp * kSub * 128;
        uint8_t* sv = sk + kHalfBytes;
        const int valid = min(kSub, p1 - (p0 + i * kStagePos + warp * kSub));
        if (valid > 0) {
            if (valid < kSub) {
                // positions past the sequence: zero K and V (the cache there is arbitrary)
                for (int r = valid; r < kSub; ++r) {
                    reinterpret_cast<uint32_t*>(sk + r * 128)[lane] = 0u;
                    reinterpret_cast<uint32_t*>(sv + r * 128)[lane] = 0u;
                }
                __syncwarp();
            }
            const uint32_t ka = smem_u32(sk), va = smem_u32(sv);

            // S = q K^T : 4 n-tiles of 8 positions
            float sacc[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
                const int r = nt * 8 + (lane & 7);
                uint32_t b[8];
                ldsm_x4(ka + sw128(r, (lane >> 3)), b[0], b[1], b[2], b[3]);
                ldsm_x4(ka + sw128(r, 4 + (lane >> 3)), b[4], b[5], b[6], b[7]);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma16816(sacc[nt], aq[kk], b[2 * kk], b[2 * kk + 1]);
            }
            // scale, mask, online softmax (rows hA -> regs 0,1 ; hB -> regs 2,3)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                if (hr == 1 && !rows_b) break;
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int pos = nt * 8 + 2 * (lane & 3) + e;
                        float v = sacc[nt][2 * hr + e] * P.scale_log2;
                        v = pos < valid ? v : -INFINITY;
                        sacc[nt][2 * hr + e] = v;
                        mx = fmaxf(mx, v);
                    }
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[hr], mx);
                const float corr = exp2f(m_run[hr] - m_new);
                float rs = 0.f;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = exp2f(sacc[nt][2 * hr + e] - m_new);
                        sacc[nt][2 * hr + e] = pv;
                        rs += pv;
                    }
                }
                rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                l_run[hr] = l_run[hr] * corr + rs;
                m_run[hr] = m_new;
#pragma unroll
                for (int nd = 0; nd < 8; ++nd) {
                    oacc[nd][2 * hr] *= corr;
                    oacc[nd][2 * hr + 1] *= corr;
                }
            }
            if (!rows_b) {
                // rows 8..15 are padding: keep their probabilities at zero
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) sacc[nt][2] = sacc[nt][3] = 0.f;
            }
            // O += P V : 2 k-steps of 16 positions x 8 n-tiles of 8 dims
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                uint32_t ap[4];
                ap[0] = pack_bf16x2(sacc[2 * kk][0], sacc[2 * kk][1]);
                ap[1] = pack_bf16x2(sacc[2 * kk][2], sacc[2 * kk][3]);
                ap[2] = pack_bf16x2(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
                ap[3] = pack_bf16x2(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
                const int mi = lane >> 3;
                const int r = kk * 16 + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                for (int nd = 0; nd < 8; nd += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(va + sw128(r, nd + (mi >> 1)), b0, b1, b2, b3);
                    mma16816(oacc[nd], ap, b0, b1);
                    mma16816(oacc[nd + 1], ap, b2, b3);
                }
            }
        }
        // release the stage; one thread refills it once every warp is done with it
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (tid == 0 && issued < nstage) {
            if (!mbar_wait(&empty[st], par, ctx.timeout_ns)) {
                report(ctx, ST_TIMEOUT, 11);
                failed = true;
            } else {
                issue(issued);
                ++issued;
            }
        }
        failed = __any_sync(0xffffffffu, failed);
        if (failed) break;
    }

    // ---- merge the four warps (fixed order) ----
    __syncthreads();  // all stages consumed: stage memory is free (no TMA pending unless failed)
    if (__syncthreads_or(failed)) {
        // drain loads still in flight (bounded): every issued stage completes its full phase
        if (tid == 0) {
            for (int i = max(0, issued - kStages); i < issued; ++i)
                (void)mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u, 10000000ull);
        }
        __syncthreads();
        task_end(ctx);
        return;
    }
    float* sm_m = reinterpret_cast<float*>(smem);   // [4][16]
    float* sm_l = sm_m + kWarps * 16;               // [4][16]
    float* sm_o = sm_l + kWarps * 16;               // [4][16][64]
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int h = hA + 8 * hr;
        if ((lane & 3) == 0) {
            sm_m[warp * 16 + h] = m_run[hr];
            sm_l[warp * 16 + h] = l_run[hr];
        }
#pragma unroll
        for (int nd = 0; nd < 8; ++nd) {
            const int d = nd * 8 + 2 * (lane & 3);
            sm_o[(warp * 16 + h) * 64 + d] = oacc[nd][2 * hr];
            sm_o[(warp * 16 + h) * 64 + d + 1] = oacc[nd][2 * hr + 1];
        }
    }
    __syncthreads();

    const size_t pair = (size_t)tl * P.nkv + kvh;
    float* pml = P.part_ml + (pair * P.S_max + s) * 32;
    float* pacc = P.part_acc + (pair * P.S_max + s) * 16 * 64;
    for (int i = tid; i < G * 64; i += kWarps * 32) {
        const int h = i >> 6, d = i & 63;
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * 16 + h]);
        float Ls = 0.f, O = 0.f;
        for (int w = 0; w < kWarps; ++w) {
            const float f = exp2f(sm_m[w * 16 + h] - M);  // exp2(-inf) = 0 for idle warps
            Ls += f * sm_l[w * 16 + h];
            O += f * sm_o[(w * 16 + h) * 64 + d];
        }
        if (S_t == 1) {
            P.o[(size_t)t * (P.nq * 64) + (size_t)(kvh * G + h) * 64 + d] =
                __float2bfloat16_rn(O / Ls);
        } else {
            pacc[h * 64 + d] = O;
            if (d == 0) {
                pml[2 * h] = M;
                pml[2 * h + 1] = Ls;
            }
        }
    }
    if (S_t > 1) {
        // ---- the last chunk of this (sequence, KV head) merges all chunks in order ----
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const uint32_t prev = atomicAdd(&P.cnt[pair], 1u);
            *sh_last = (prev == (uint32_t)S_t - 1) ? 1 : 0;
            if (*sh_last) P.cnt[pair] = 0;
        }
        __syncthreads();
        if (*sh_last) {
            __threadfence();
            const float* bml = P.part_ml + pair * P.S_max * 32;
            const float* bacc = P.part_acc + pair * P.S_max * 16 * 64;
            for (int i = tid; i < G * 64; i += kWarps * 32) {
                const int h = i >> 6, d = i & 63;
                float M = -INFINITY;
                for (int c = 0; c < S_t; ++c) M = fmaxf(M, __ldcg(bml + c * 32 + 2 * h));
                float Ls = 0.f, O = 0.f;
                for (int c = 0; c < S_t; ++c) {
                    const float f = exp2f(__ldcg(bml + c * 32 + 2 * h) - M);
                    Ls += f * __ldcg(bml + c * 32 + 2 * h + 1);
                    O += f * __ldcg(bacc + (c * 16 + h) * 64 + d);
                }
                P.o[(size_t)t * (P.nq * 64) + (size_t)(kvh * G + h) * 64 + d] =
                    __float2bfloat16_rn(O / Ls);
            }
        }
    }
    task_end(ctx);
}

}  // namespace

int enqueue_attention(Launcher& L, const AttnProblem& p, const KCtx& c) {
    dim3 grid(p.S_max, p.nkv, p.nrows), block(kWarps * 32);
    size_t smem = kStages * kStageBytes + 1024 + 256;  // merge scratch reuses the stages
    void* args[] = {(void*)&p, (void*)&c};
    return L.launch((const void*)attn_decode_kernel, grid, block, smem, args);
}

}  // namespace sgp
