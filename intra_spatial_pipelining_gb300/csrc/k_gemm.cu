// Projections of the decode layer: QKV (+ KV-cache append), output projection (+ residual),
// grouped expert gate/up (+ SwiGLU) and grouped expert down.
//
// Decode gives few tokens per weight matrix (64 per layer, 16-64 per expert slot), so the
// contraction is "swap-AB": the weight tile is the MMA's M = 128 operand and the tokens are
// its N (16..256) operand.  Two kernels per projection:
//   gemm_tc_kernel   persistent, one work unit = (group, 128-row weight tile, K segment):
//                    weights stream HBM -> shared memory through a TMA ring (128-byte
//                    swizzle), one elected lane issues tcgen05.mma into a double-buffered
//                    TMEM accumulator, and the tile leaves through shared memory -- with the
//                    epilogue applied when the K split is 1, else as one TMA bulk store per
//                    chunk into a partial-sum buffer.  No cross-CTA protocol.
//   gemm_finish_kernel  every thread owns 4 consecutive outputs of one token: it sums the
//                    K segments in segment order (fixed, so results never depend on the
//                    grid or the token count) and applies the epilogue with 16-byte loads.
//                    (The expert-down projection has none: the combine sums its segments.)
#include <algorithm>

#include "kernels.h"

namespace sgp {

namespace {

constexpr int kThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kRunAheadL2 = 8;  // weight stages a dense producer pulls into L2 before its wait

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// named barrier of the 4 epilogue warps
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// same barrier, returning the OR of `v` over the 128 epilogue threads (uniform decision)
__device__ __forceinline__ bool epi_bar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Rotates 4 consecutive features of one head (head-local index hf, a multiple of 4) by the
// RoPE angles at position pos; p holds the pair partners (features hf +- 32).  The angle
// pos * w_i is formed in float-float (w_i = hi + lo from the host) and reduced modulo 2 pi
// with a two-constant Cody-Waite split before sincosf, so positions up to 2^24 keep
// about 1e-6 rad of accuracy.
__device__ __forceinline__ void rope_rotate(float4& v, const float4& p, int hf, int pos,
                                            const EpiArgs& e) {
    const float x[4] = {v.x, v.y, v.z, v.w}, y[4] = {p.x, p.y, p.z, p.w};
    float o[4];
    const bool first = hf < 32;
    const float fp = (float)pos;
    constexpr float kTwoPiHi = 6.28318548202514648f;      // nearest float to 2 pi
    constexpr float kTwoPiLo = -1.7484555314695172e-07f;  // 2 pi - kTwoPiHi
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int i = (hf + c) & 31;
        const float hi = e.rope_fhi[i], lo = e.rope_flo[i];
        const float a = fp * hi;
        const float a_err = fmaf(fp, hi, -a) + fp * lo;   // a + a_err = pos * w_i
        const float k = rintf(a * 0.159154943091895336f);   // turns
        const float r = (fmaf(-k, kTwoPiHi, a) + fmaf(-k, kTwoPiLo, 0.f)) + a_err;
        float sn, cs;
        sincosf(r, &sn, &cs);
        o[c] = first ? fmaf(x[c], cs, -y[c] * sn) : fmaf(y[c], sn, x[c] * cs);
    }
    v = make_float4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------------------------------
// Epilogue stores shared by the finishing pass and the GEMM's own epilogue (K split 1).
// v holds 4 consecutive output features f0..f0+3 of token row trow (RoPE already applied).
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void store_out4(const EpiArgs& e, const KCtx& ctx, int mode, int trow,
                                           int f0, float4 v) {
    if (mode == EPI_F32) {
        *reinterpret_cast<float4*>(e.out_f32 + (size_t)trow * e.ld + f0) = v;
        return;
    }
    if (mode == EPI_RESID) {
        const uint2 rr = *reinterpret_cast<const uint2*>(e.resid + (size_t)trow * e.ld + f0);
        const float2 r01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rr.x));
        const float2 r23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rr.y));
        v.x += r01.x;
        v.y += r01.y;
        v.z += r23.x;
        v.w += r23.y;
    }
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    bf16* dst;
    if (mode == EPI_RESID) {
        dst = e.out + (size_t)trow * e.ld + f0;
    } else if (f0 < e.q_width) {  // EPI_QKV: query heads
        dst = e.q + (size_t)trow * e.q_width + f0;
    } else {                      // EPI_QKV: append k / v at slot kv_len - 1
        const int r = f0 - e.q_width;
        const int which = r / (e.nkv * e.d);
        const int kh = (r / e.d) % e.nkv;
        const int pos = e.kv_len[trow] - 1;
        if (pos < 0 || pos >= e.cap) {
            report(ctx, ST_BOUNDS, (uint32_t)pos);
            return;
        }
        bf16* cache = which == 0 ? e.kc : e.vc;
        dst = cache + (((size_t)trow * e.nkv + kh) * e.cap + pos) * e.d + (r % e.d);
    }
    *reinterpret_cast<uint2*>(dst) = o;
}

__device__ __forceinline__ void store_swiglu4(const EpiArgs& e, int trow, int i0, float4 g,
                                              float4 up) {
    uint2 o;
    o.x = pack_bf16x2(silu_f(g.x) * up.x, silu_f(g.y) * up.y);
    o.y = pack_bf16x2(silu_f(g.z) * up.z, silu_f(g.w) * up.w);
    *reinterpret_cast<uint2*>(e.out + (size_t)trow * e.ld + i0) = o;
}

// One work unit = (group, 128-row weight tile, K segment) and its token range, covered in
// npass passes of up to n_cap tokens; the last pass also carries `tail` more rows (0: none)
// when the rows past its end fit tail_cap.
struct Unit {
    int g, mt, ks, kb0, nk, n, npass, tail, tma_r0, lr0;
};

__device__ __forceinline__ Unit unit_info(const GemmProblem& P, int u, const KCtx& c) {
    Unit x;
    const int per_group = P.m_tiles * P.ksplit;
    x.g = u / per_group;
    const int rem = u % per_group;
    x.mt = rem / P.ksplit;
    x.ks = rem % P.ksplit;
    if (P.serpentine) x.g = P.n_groups - 1 - x.g;
    // K segment = stage blocks [sb0, sb1); k-blocks beyond K are zero-filled by the loads
    const int sb0 = (x.ks * P.n_sb) / P.ksplit;
    x.kb0 = sb0 * P.kps;
    x.nk = ((x.ks + 1) * P.n_sb) / P.ksplit - sb0;  // stage blocks of this segment
    if (P.group_offsets != nullptr) {
        x.tma_r0 = P.group_offsets[x.g];
        x.n = P.group_offsets[x.g + 1] - x.tma_r0;
        x.lr0 = x.tma_r0;
    } else {
        x.tma_r0 = 0;
        x.n = P.nrows;
        x.lr0 = 0;
    }
    if (x.lr0 < 0 || x.n < 0 || x.lr0 + x.n > P.R) {
        if (threadIdx.x == 0) report(c, ST_BOUNDS, (uint32_t)(x.lr0 + x.n));
        x.n = 0;
    }
    if (x.nk <= 0) x.n = 0;
    const int n_pad = (x.n + 15) & ~15;
    x.npass = (n_pad + P.n_cap - 1) / P.n_cap;
    x.tail = 0;
    if (P.tail_cap > 0 && x.npass >= 2 && n_pad - (x.npass - 1) * P.n_cap <= P.tail_cap) {
        x.tail = n_pad - (x.npass - 1) * P.n_cap;
        x.npass -= 1;
    }
    return x;
}

// Persistent: CTA b processes units b, b + gridDim.x, ... in that order; every role walks the
// same job sequence (unit, pass), so the ring and TMEM phases line up without messages.
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ GemmProblem P, const KCtx ctx) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = P.stages;
    const int stage_a = P.kps * 128 * 128;      // A: kps k-blocks of 128 rows x 64 bf16
    const int stage_b = P.kps * P.n_cap * 128;  // B: kps k-blocks of n_cap rows
    const int stage_t = P.kps * P.tail_cap * 128;  // tail rows (after B)
    const int stage_bytes = stage_a + stage_b + stage_t;
    float* Ts = reinterpret_cast<float*>(smem + (size_t)S * stage_bytes);  // [n_cap][128]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + P.ring_bytes);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;   // [2] accumulator ready
    uint64_t* tempty = tfull + 2;  // [2] accumulator drained
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    int* sh_err = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    griddep_launch();
    uint32_t acc_cols = 32;
    while (acc_cols < (uint32_t)P.n_cap) acc_cols <<= 1;
    // accumulators: two buffers (the epilogue drains one while the next job accumulates into
    // the other); with tail passes one buffer of the main and the tail accumulator side by
    // side (the tail's columns follow the main ones)
    const uint32_t nbuf = P.tail_cap > 0 ? 1u : 2u;
    uint32_t tmem_cols = 2 * acc_cols;
    if (P.tail_cap > 0) {
        tmem_cols = 32;
        while (tmem_cols < acc_cols + (uint32_t)P.tail_cap) tmem_cols <<= 1;
    }

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        *sh_err = 0;
        fence_barrier_init();
        prefetch_tensormap(&P.tmA);
        prefetch_tensormap(&P.tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Only the producer warp of a dense problem may run ahead of the previous kernel: its
    // elected lane streams constant weights into the ring before it waits.  The decision is
    // per warp: were the other lanes to wait here, the producer lane would be held at the
    // warp's reconvergence point until the previous kernel completes.  A grouped problem's
    // token ranges come from the previous kernel, so there everyone waits now.
    const bool run_ahead = warp == 0 && P.group_offsets == nullptr;
    if (warp == 0 && lane == 0 && !run_ahead) {
        // grouped problem: which tokens a unit covers is known only after the previous kernel,
        // but its weight tiles are not -- pull the first ring's worth of them into L2 while
        // that kernel drains (a plain wait when the launch is not programmatic)
        int q = 0;
        const int per_group = P.m_tiles * P.ksplit;
        for (int u = blockIdx.x; u < P.n_units && q < S; u += gridDim.x) {
            int g = u / per_group;
            const int rem = u % per_group, mt = rem / P.ksplit, ks = rem % P.ksplit;
            if (P.serpentine) g = P.n_groups - 1 - g;
            const int sb0 = (ks * P.n_sb) / P.ksplit, nk = ((ks + 1) * P.n_sb) / P.ksplit - sb0;
            const int rowA1 = g * P.rows_per_group + mt * P.a_tile_stride;
            for (int i = 0; i < nk && q < S; ++i, ++q) {
                const int kb = (sb0 + i) * P.kps;
                if (P.a_4d) tma_prefetch_4d(&P.tmA, 0, rowA1, 0, kb);
                else tma_prefetch_3d(&P.tmA, 0, rowA1, kb);
            }
        }
    }
    if (!run_ahead) griddep_wait();
    task_begin(ctx, 32);

    if (warp == 0) {
        // ================= TMA producer =================
        // One elected lane of the converged warp walks the whole job sequence while the other
        // lanes wait at the warp barrier below (issue from a lane whose warp-mates sit at the
        // CTA barrier is measurably slower).
        if (elect_one()) {
            // a weight tile read again by a later token pass of the same unit (or by a later
            // microbatch) is kept in L2; its last read lets it go first
            const uint64_t pol_keep = policy_evict_last();
            const uint64_t pol_drop = P.keep_weights ? pol_keep : policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            uint32_t it = 0;
            uint32_t issued_mask = 0, issued_par = 0;
            bool dropped = false;
            // activation loads deferred until the previous kernel has completed
            bool waited = !run_ahead;
            int pend_n = 0, pend_s[8], pend_row[8], pend_kb[8];
            for (int u = blockIdx.x; u < P.n_units && !*(volatile int*)sh_err; u += gridDim.x) {
                const Unit x = unit_info(P, u, ctx);
                const int rowA1 = x.g * P.rows_per_group + x.mt * P.a_tile_stride;
                for (int pass = 0; pass < x.npass; ++pass) {
                    const int c0 = pass * P.n_cap;
                    const uint64_t pol_w = pass + 1 < x.npass ? pol_keep : pol_drop;
                    const bool with_tail = x.tail > 0 && pass + 1 == x.npass;
                    const uint32_t tx = (uint32_t)(stage_a + stage_b + (with_tail ? stage_t : 0));
                    for (int i = 0; i < x.nk; ++i, ++it) {
                        const int s = it % S;
                        const uint32_t j = it / S;
                        if (!waited && j > 0) {
                            // every stage holds weights; pull the weight tiles that come next
                            // into L2 as well.  The previous kernel must be complete before
                            // the deferred activation loads (and any reuse) go out.
                            int q = 0;
                            for (int u2 = u; u2 < P.n_units && q < kRunAheadL2; u2 += gridDim.x) {
                                const Unit y = unit_info(P, u2, ctx);
                                const int rowA2 = y.g * P.rows_per_group + y.mt * P.a_tile_stride;
                                for (int i2 = u2 == u ? i : 0; i2 < y.nk && q < kRunAheadL2; ++i2, ++q) {
                                    const int kb2 = y.kb0 + i2 * P.kps;
                                    if (P.a_4d) tma_prefetch_4d(&P.tmA, 0, rowA2, 0, kb2);
                                    else tma_prefetch_3d(&P.tmA, 0, rowA2, kb2);
                                }
                            }
                            griddep_wait();
                            waited = true;
                            for (int q = 0; q < pend_n; ++q)
                                tma_load_3d(smem + (size_t)pend_s[q] * stage_bytes + stage_a,
                                            &P.tmB, &full[pend_s[q]], 0, pend_row[q], pend_kb[q],
                                            pol_x);
                        }
                        if (j > 0 && !mbar_wait(&empty[s], (j - 1) & 1, ctx.timeout_ns)) {
                            report(ctx, ST_TIMEOUT, 1);
                            atomicExch(sh_err, 1);
                            break;
                        }
                        if ((ctx.fault & FAULT_DROP_TMA) && blockIdx.x == 0 && !dropped) {
                            dropped = true;  // test-only: this stage never fills
                            continue;
                        }
                        uint8_t* sa = smem + (size_t)s * stage_bytes;
                        uint8_t* sb = sa + stage_a;
                        const int kb = x.kb0 + i * P.kps;
                        mbar_arrive_expect_tx(&full[s], tx);
                        if (P.a_4d)
                            tma_load_4d(sa, &P.tmA, &full[s], 0, rowA1, 0, kb, pol_w);
                        else
                            tma_load_3d(sa, &P.tmA, &full[s], 0, rowA1, kb, pol_w);
                        if (!waited) {  // first pass over the ring: activations wait
                            pend_s[pend_n] = s;
                            pend_row[pend_n] = x.tma_r0 + c0;
                            pend_kb[pend_n] = kb;
                            ++pend_n;
                        } else {
                            tma_load_3d(sb, &P.tmB, &full[s], 0, x.tma_r0 + c0, kb, pol_x);
                        }
                        if (with_tail)  // grouped problems only: never deferred
                            tma_load_3d(sb + stage_b, &P.tmB2, &full[s], 0, x.tma_r0 + c0 + P.n_cap,
                                        kb, pol_x);
                        issued_mask |= 1u << s;
                        issued_par = (issued_par & ~(1u << s)) | ((j & 1u) << s);
                    }
                    if (*(volatile int*)sh_err) break;
                }
            }
            if (!waited) {
                griddep_wait();
                for (int q = 0; q < pend_n; ++q)
                    tma_load_3d(smem + (size_t)pend_s[q] * stage_bytes + stage_a, &P.tmB,
                                &full[pend_s[q]], 0, pend_row[q], pend_kb[q], pol_x);
            }
            if (*(volatile int*)sh_err) {
                // drain loads still in flight into this CTA's shared memory (bounded)
                for (int s = 0; s < S; ++s)
                    if (issued_mask & (1u << s))
                        (void)mbar_wait(&full[s], (issued_par >> s) & 1u, 10000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        // One elected lane issues every MMA and commit (single-thread semantics); see above.
        if (elect_one()) {
            uint32_t it = 0, job = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < P.n_units && ok; u += gridDim.x) {
                const Unit x = unit_info(P, u, ctx);
                const int n_pad = (x.n + 15) & ~15;
                for (int pass = 0; pass < x.npass && ok; ++pass, ++job) {
                    const int np = min(P.n_cap, n_pad - pass * P.n_cap);
                    const bool with_tail = x.tail > 0 && pass + 1 == x.npass;
                    const uint32_t b = job % nbuf, jb = job / nbuf;
                    if (jb > 0 && !mbar_wait(&tempty[b], (jb - 1) & 1u, ctx.timeout_ns)) {
                        report(ctx, ST_TIMEOUT, 5);
                        atomicExch(sh_err, 1);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acc = tmem + b * acc_cols;
                    const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)np);
                    const uint32_t idesc_t = idesc_bf16_f32(128, (uint32_t)max(16, x.tail));
                    for (int i = 0; i < x.nk; ++i, ++it) {
                        const int s = it % S;
                        const uint32_t j = it / S;
                        if (!mbar_wait(&full[s], j & 1, ctx.timeout_ns)) {
                            report(ctx, ST_TIMEOUT, 2);
                            atomicExch(sh_err, 1);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
                        const uint32_t sb = sa + stage_a;
#pragma unroll
                        for (int kk = 0; kk < kGemmKpsMax; ++kk)
                            if (kk < P.kps) {
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    tc_mma_bf16(acc, smem_desc_sw128(sa + kk * 16384 + 32 * k),
                                                smem_desc_sw128(sb + kk * (P.n_cap * 128) + 32 * k),
                                                idesc, (i > 0 || kk > 0 || k > 0) ? 1u : 0u);
                                    // the tail rows take the same k steps in the same order
                                    if (with_tail)
                                        tc_mma_bf16(acc + acc_cols,
                                                    smem_desc_sw128(sa + kk * 16384 + 32 * k),
                                                    smem_desc_sw128(sb + stage_b + kk * (P.tail_cap * 128) + 32 * k),
                                                    idesc_t, (i > 0 || kk > 0 || k > 0) ? 1u : 0u);
                                }
                            }
                        tc_commit(&empty[s]);
                    }
                    if (ok) tc_commit(&tfull[b]);
                }
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue: TMEM -> shared -> one bulk store per job =================
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const int row = q * 32 + lane;
        const bool issuer = (warp == 2 && lane == 0);
        uint32_t job = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < P.n_units && ok; u += gridDim.x) {
            const Unit x = unit_info(P, u, ctx);
            const int n_pad = (x.n + 15) & ~15;
            for (int pass = 0; pass < x.npass; ++pass, ++job) {
                const uint32_t b = job % nbuf, jb = job / nbuf;
                const bool with_tail = x.tail > 0 && pass + 1 == x.npass;
                const bool w = mbar_wait(&tfull[b], jb & 1u, ctx.timeout_ns);
                if (!w) {
                    report(ctx, ST_TIMEOUT, 3);
                    atomicExch(sh_err, 1);
                }
                // the previous job's bulk store must have finished reading Ts
                if (issuer) bulk_wait_read();
                // all four epilogue warps take the same decision
                if (epi_bar_or(!w || *(volatile int*)sh_err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // part 0: the pass's own accumulator; part 1: the tail rows that follow it
                for (int part = 0; part < (with_tail ? 2 : 1); ++part) {
                    const int c0 = pass * P.n_cap + part * P.n_cap;
                    const int np = part ? x.tail : min(P.n_cap, n_pad - c0);
                    const uint32_t tbase = tmem + (part ? acc_cols : b * acc_cols) +
                                           ((uint32_t)(q * 32) << 16);
                    const int nv = min(np, x.n - c0);
                    const bool last_part = part + 1 == (with_tail ? 2 : 1);
                    // the accumulator leaves TMEM in chunks of ts_rows tokens through Ts
                    for (int ch = 0; ch < np; ch += P.ts_rows) {
                        const int cn = min(P.ts_rows, np - ch);
                        if (ch > 0 || part > 0) {
                            // the previous chunk's readers (bulk store / epilogue) are done with Ts
                            if (issuer) bulk_wait_read();
                            epi_bar();
                        }
                        for (int cc = 0; cc < cn; cc += 16) {
                            uint32_t v[16];
                            tmem_ld_x16(tbase + (uint32_t)(ch + cc), v);
                            tmem_ld_wait();
#pragma unroll
                            for (int t = 0; t < 16; ++t) Ts[(cc + t) * 128 + row] = __uint_as_float(v[t]);
                        }
                        if (last_part && ch + P.ts_rows >= np) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[b]);  // the accumulator may be reused
                        }
                        const int cv = min(cn, nv - ch);  // valid tokens of this chunk
                        if (P.fused_epi) {
                            // K split 1: the tile is the final sum; apply the epilogue from Ts
                            // (the next chunk's or job's barrier keeps Ts until every warp is done)
                            epi_bar();
                            const EpiArgs& e = P.epi;
                            const int ew = warp - 2;  // 0..3
                            const int prow0 = x.lr0 + c0 + ch;  // partial-row numbering of token 0
                            if (e.mode == EPI_SWIGLU) {
                                const int h = lane >> 4, q4 = lane & 15;
                                const int i0 = x.mt * 64 + 4 * q4;
                                for (int t = 2 * ew + h; t < cv; t += 8) {
                                    if (i0 < e.n_out) {
                                        const float4 g = *reinterpret_cast<const float4*>(Ts + t * 128 + 4 * q4);
                                        const float4 up = *reinterpret_cast<const float4*>(Ts + t * 128 + 64 + 4 * q4);
                                        store_swiglu4(e, P.out_row0 + prow0 + t, i0, g, up);
                                    }
                                }
                            } else {
                                const int f0 = x.mt * 128 + 4 * lane;
                                for (int t = ew; t < cv; t += 4) {
                                    const int trow = P.out_row0 + prow0 + t;
                                    float4 v = *reinterpret_cast<const float4*>(Ts + t * 128 + 4 * lane);
                                    if (e.mode == EPI_QKV && e.rope_theta > 0.f) {
                                        // pair partner (feature +-32 of the same head): lane ^ 8
                                        const float4 pv = *reinterpret_cast<const float4*>(Ts + t * 128 + 4 * (lane ^ 8));
                                        if (f0 < e.n_out && f0 < e.q_width + e.nkv * e.d)
                                            rope_rotate(v, pv, f0 & 63, e.kv_len[trow] - 1, e);
                                    }
                                    if (f0 < e.n_out) store_out4(e, ctx, e.mode, trow, f0, v);
                                }
                            }
                        } else if (cv > 0) {
                            fence_proxy_async();
                            epi_bar();
                            if (issuer) {
                                bulk_store(P.partial + (((size_t)x.mt * P.ksplit + x.ks) * P.R + x.lr0 + c0 + ch) * 128,
                                           Ts, (uint32_t)cv * 512u);
                                bulk_commit();
                            }
                        } else {
                            epi_bar();
                        }
                    }
                }
            }
        }
        if (issuer) bulk_wait_all();  // partial tiles complete before the CTA finishes
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
    task_end(ctx);
}

// ---------------------------------------------------------------------------------------
// K-segment reduction + fused epilogue: one thread = 4 consecutive outputs of one token.  The
// K-segment loads are issued before they are summed (in segment order).
// ---------------------------------------------------------------------------------------
// U loads in flight per thread and sum; the kernel is instantiated for U = 4 and 8 so that a
// small K split does not pay the registers (and the occupancy) of a large one.
template <int U>
__device__ __forceinline__ float4 sum_segments(const float* p, size_t sstride, int ks) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ks; s0 += U) {
        float4 v[U];
#pragma unroll
        for (int i = 0; i < U; ++i)
            if (s0 + i < ks) v[i] = __ldcg(reinterpret_cast<const float4*>(p + (s0 + i) * sstride));
#pragma unroll
        for (int i = 0; i < U; ++i)
            if (s0 + i < ks) {
                acc.x += v[i].x;
                acc.y += v[i].y;
                acc.z += v[i].z;
                acc.w += v[i].w;
            }
    }
    return acc;
}

// Instantiated per epilogue (MODE) so that each variant keeps only its own registers.
template <int U, int MODE>
__global__ void __launch_bounds__(256, U <= 4 ? 4 : 2)
    gemm_finish_kernel(const FinishProblem P, const KCtx ctx) {
    griddep_launch();
    griddep_wait();
    task_begin(ctx);
    const EpiArgs& e = P.epi;
    constexpr bool swiglu = MODE == EPI_SWIGLU;
    const int per_tok = swiglu ? 16 : 32;         // 4-output groups per (tile, token)
    const int total = P.m_tiles * P.rows * per_tok;
    const size_t sstride = (size_t)P.R * 128;     // next K segment
    for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < total; u += gridDim.x * blockDim.x) {
        const int q4 = u % per_tok;
        const int lr = (u / per_tok) % P.rows;
        const int mt = u / (per_tok * P.rows);
        const float* base = P.partial + ((size_t)mt * P.ksplit * P.R + lr) * 128;
        const int trow = P.out_row0 + lr;
        if constexpr (swiglu) {
            const int i0 = mt * 64 + 4 * q4;
            if (i0 >= e.n_out) continue;
            const float4 g = sum_segments<U>(base + 4 * q4, sstride, P.ksplit);
            const float4 up = sum_segments<U>(base + 64 + 4 * q4, sstride, P.ksplit);
            store_swiglu4(e, trow, i0, g, up);
            continue;
        }
        const int f0 = mt * 128 + 4 * q4;  // first of the 4 output features
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (f0 < e.n_out) v = sum_segments<U>(base + 4 * q4, sstride, P.ksplit);
        if constexpr (MODE == EPI_QKV) {
            // RoPE on q and k: the pair partner (feature +-32 of the same head) sits in lane
            // q4 ^ 8 of this warp (32 lanes per token row, loop stride a multiple of 32), so
            // the whole warp exchanges before any lane leaves the iteration
            if (e.rope_theta > 0.f) {
                float4 pv;
                pv.x = __shfl_xor_sync(0xffffffffu, v.x, 8);
                pv.y = __shfl_xor_sync(0xffffffffu, v.y, 8);
                pv.z = __shfl_xor_sync(0xffffffffu, v.z, 8);
                pv.w = __shfl_xor_sync(0xffffffffu, v.w, 8);
                if (f0 < e.n_out && f0 < e.q_width + e.nkv * e.d)
                    rope_rotate(v, pv, f0 & 63, e.kv_len[trow] - 1, e);
            }
        }
        if (f0 >= e.n_out) continue;
        store_out4(e, ctx, MODE, trow, f0, v);
    }
    task_end(ctx);
}

// ---------------------------------------------------------------------------------------
// GEMV path (fewer than gemv_max_tokens tokens per weight matrix): a skinny product whose
// weights stream straight from HBM into registers.  A warp owns a tile of 16 weight rows --
// 16 output features, or 8 SwiGLU features as 8 gate rows over 8 up rows -- and one eighth of
// K; the CTA's 8 warps cover all of K and add their partial tiles in warp order through
// shared memory.  The per-lane product is a warp-level bf16 MMA (m16n8k16, fp32 accumulate)
// over 8 tokens per n-tile, which does the K reduction without shuffles.  Its operands come
// straight from 16-byte loads: in every 32-wide K block, lane (g, t) loads K positions
// [8t, 8t + 8) of weight rows g and g + 8 and of token g's activation row, and the two MMAs
// of the block take positions 8t..8t+3 and 8t+4..8t+7 as the fragment columns
// {2t, 2t+1, 2t+8, 2t+9} -- the same permutation of K for both operands, so each MMA still
// sums products of matching elements.  kGemvU blocks of loads (4 x 16 bytes per lane each)
// are issued before their MMAs.  A token's result never depends on the other tokens.
// ---------------------------------------------------------------------------------------
constexpr int kGemvWarps = 8;  // K split of a tile (one warp per part)
constexpr int kGemvU = 4;      // 32-wide K blocks whose loads are in flight together

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void gemv_store(const EpiArgs& e, const KCtx& c, int f, int trow,
                                           float v) {
    if (f >= e.n_out) return;
    switch (e.mode) {
        case EPI_QKV: {
            if (f < e.q_width) {
                e.q[(size_t)trow * e.q_width + f] = __float2bfloat16_rn(v);
            } else {
                const int r = f - e.q_width;
                const int which = r / (e.nkv * e.d);
                const int kh = (r / e.d) % e.nkv;
                const int pos = e.kv_len[trow] - 1;
                if (pos < 0 || pos >= e.cap) {
                    report(c, ST_BOUNDS, (uint32_t)pos);
                    return;
                }
                bf16* cache = which == 0 ? e.kc : e.vc;
                cache[(((size_t)trow * e.nkv + kh) * e.cap + pos) * e.d + (r % e.d)] =
                    __float2bfloat16_rn(v);
            }
            break;
        }
        case EPI_RESID: {
            const size_t o = (size_t)trow * e.ld + f;
            e.out[o] = __float2bfloat16_rn(__bfloat162float(e.resid[o]) + v);
            break;
        }
        case EPI_F32:
            e.out_f32[(size_t)trow * e.ld + f] = v;
            break;
        default:
            break;
    }
}

// NT n-tiles of 8 tokens per pass (1: up to 8 tokens, 2: up to 16)
template <int NT>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_kernel(const GemvProblem P, const KCtx ctx) {
    griddep_launch();
    griddep_wait();
    task_begin(ctx);
    __shared__ float red[kGemvWarps][32][4 * NT];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = lane >> 2, ti = lane & 3;   // fragment row group / column pair
    const int g = blockIdx.y;
    // the tile's weight rows g and g + 8 of this lane, and the features they feed
    int row_lo, row_hi, f_lo, f_hi;
    if (P.swiglu) {
        f_lo = f_hi = blockIdx.x * 8 + gi;             // gate row over up row of one feature
        row_lo = f_lo;
        row_hi = f_lo + P.up_off;
    } else {
        f_lo = blockIdx.x * 16 + gi;
        f_hi = f_lo + 8;
        row_lo = f_lo;
        row_hi = f_hi;
    }
    const bool ok_lo = f_lo < P.n_out, ok_hi = f_hi < P.n_out;
    const uint4* wlo = reinterpret_cast<const uint4*>(P.W + ((size_t)g * P.rows_per_group + row_lo) * P.K);
    const uint4* whi = reinterpret_cast<const uint4*>(P.W + ((size_t)g * P.rows_per_group + row_hi) * P.K);
    int r0, n;
    if (P.group_offsets != nullptr) {
        r0 = P.group_offsets[g];
        n = P.group_offsets[g + 1] - r0;
    } else {
        r0 = P.row0;
        n = P.nrows;
    }
    const int nkb = P.K >> 5;                                   // 32-wide K blocks
    const int kb0 = warp * nkb / kGemvWarps, kb1 = (warp + 1) * nkb / kGemvWarps;
    const uint4 z4 = make_uint4(0, 0, 0, 0);
    for (int t0 = 0; t0 < n; t0 += 8 * NT) {
        float acc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        const uint4* xr[NT];
        bool xok[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int t = t0 + 8 * j + gi;                      // this lane's token of n-tile j
            xok[j] = t < n;
            xr[j] = reinterpret_cast<const uint4*>(P.X + (size_t)(r0 + (xok[j] ? t : 0)) * P.K);
        }
        for (int kb = kb0; kb < kb1; kb += kGemvU) {
            uint4 alo[kGemvU], ahi[kGemvU], b[kGemvU][NT];
#pragma unroll
            for (int u = 0; u < kGemvU; ++u) {
                const bool in = kb + u < kb1;
                const int c = (kb + u) * 4 + ti;                // 16-byte chunk of the row
                alo[u] = (in && ok_lo) ? __ldg(wlo + c) : z4;
                ahi[u] = (in && ok_hi) ? __ldg(whi + c) : z4;
#pragma unroll
                for (int j = 0; j < NT; ++j) b[u][j] = (in && xok[j]) ? __ldg(xr[j] + c) : z4;
            }
#pragma unroll
            for (int u = 0; u < kGemvU; ++u) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    mma16816(acc[j], alo[u].x, ahi[u].x, alo[u].y, ahi[u].y, b[u][j].x, b[u][j].y);
                    mma16816(acc[j], alo[u].z, ahi[u].z, alo[u].w, ahi[u].w, b[u][j].z, b[u][j].w);
                }
            }
        }
        // the 8 K parts of the tile, added in warp order
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp][lane][4 * j + i] = acc[j][i];
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[i] = red[0][lane][4 * j + i];
#pragma unroll
                    for (int w = 1; w < kGemvWarps; ++w) v[i] += red[w][lane][4 * j + i];
                }
                // fragment: rows gi (v0, v1) and gi + 8 (v2, v3), tokens 2 ti and 2 ti + 1
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int t = t0 + 8 * j + 2 * ti + c;
                    if (t >= n) continue;
                    const int trow = r0 + t;
                    if (P.swiglu) {
                        if (ok_lo)
                            P.epi.out[(size_t)trow * P.epi.ld + f_lo] =
                                __float2bfloat16_rn(silu_f(v[c]) * v[2 + c]);
                    } else {
                        if (ok_lo) gemv_store(P.epi, ctx, f_lo, trow, v[c]);
                        if (ok_hi) gemv_store(P.epi, ctx, f_hi, trow, v[2 + c]);
                    }
                }
            }
        }
        __syncthreads();  // red is reused by the next token pass
    }
    task_end(ctx);
}

}  // namespace

size_t gemm_tc_ring_bytes(int n_cap, int stages, int kps, int tail_cap, int ts_rows) {
    // stage ring, then the accumulator staging area [min(n_cap, ts_rows)][128] fp32
    return (size_t)stages * kps * (128 * 128 + (n_cap + tail_cap) * 128) +
           (size_t)std::min(n_cap, ts_rows) * 512;
}

size_t gemm_tc_smem_bytes(int n_cap, int stages, int kps, int tail_cap, int ts_rows) {
    return gemm_tc_ring_bytes(n_cap, stages, kps, tail_cap, ts_rows) + 1024 + 256;
}

int enqueue_gemm_tc(Launcher& L, const GemmProblem& p, const KCtx& c) {
    dim3 grid(std::max(1, std::min(p.n_units, p.grid))), block(kThreads);
    // the tail accumulator sits beside a single main buffer in the 512 TMEM columns
    if ((p.kps != 1 && p.kps != 2) || (p.ts_rows != 32 && p.ts_rows != 64) ||
        p.tail_cap < 0 || (p.tail_cap & 15) || p.tail_cap + p.n_cap > 512 ||
        (p.tail_cap > 0 && p.group_offsets == nullptr) ||
        (size_t)p.ring_bytes != gemm_tc_ring_bytes(p.n_cap, p.stages, p.kps, p.tail_cap, p.ts_rows))
        return (int)cudaErrorInvalidValue;
    void* args[] = {(void*)&p, (void*)&c};
    return L.launch((const void*)gemm_tc_kernel, grid, block,
                    gemm_tc_smem_bytes(p.n_cap, p.stages, p.kps, p.tail_cap, p.ts_rows), args, true);
}

int enqueue_gemm_finish(Launcher& L, const FinishProblem& p, const KCtx& c) {
    const int per_tok = p.epi.mode == EPI_SWIGLU ? 16 : 32;
    const long total = (long)p.m_tiles * p.rows * per_tok;
    const int blocks = (int)std::min<long>((total + 255) / 256, 4096);
    void* args[] = {(void*)&p, (void*)&c};
    const bool small = p.ksplit <= 4;
    const void* f = nullptr;
    switch (p.epi.mode) {
        case EPI_QKV:
            f = small ? (const void*)gemm_finish_kernel<4, EPI_QKV> : (const void*)gemm_finish_kernel<8, EPI_QKV>;
            break;
        case EPI_RESID:
            f = small ? (const void*)gemm_finish_kernel<4, EPI_RESID>
                      : (const void*)gemm_finish_kernel<8, EPI_RESID>;
            break;
        case EPI_SWIGLU:
            f = small ? (const void*)gemm_finish_kernel<4, EPI_SWIGLU>
                      : (const void*)gemm_finish_kernel<8, EPI_SWIGLU>;
            break;
        default:
            f = small ? (const void*)gemm_finish_kernel<4, EPI_F32> : (const void*)gemm_finish_kernel<8, EPI_F32>;
            break;
    }
    return L.launch(f, dim3(std::max(1, blocks)), dim3(256), 0, args, true);
}

int enqueue_gemv(Launcher& L, const GemvProblem& p, const KCtx& c) {
    if (p.K % 32) return (int)cudaErrorInvalidValue;  // 32-wide K blocks
    const int per_tile = p.swiglu ? 8 : 16;          // output features per 16-row tile
    dim3 grid((p.n_out + per_tile - 1) / per_tile, p.n_groups), block(kGemvWarps * 32);
    void* args[] = {(void*)&p, (void*)&c};
    // two n-tiles per pass when a matrix may see more than 8 tokens
    const int most = p.group_offsets ? 16 : p.nrows;
    return L.launch(most > 8 ? (const void*)gemv_kernel<2> : (const void*)gemv_kernel<1>, grid,
                    block, 0, args);
}

}  // namespace sgp
