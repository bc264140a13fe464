// attn_bwd.cu - exact attention backward for sm_103a (TMA + tcgen05 + TMEM).
//
// Three kernels, launched in this order on the caller's stream:
//  1. preprocess: D_i = sum_j P_ij dP_ij in fp32 and dq_accum := 0
//     (wonbeomjang.kr FlashAttention-2 review, "Backward Pass": D is the
//     softmax-gradient row term, computed ahead of the main loop);
//  2. main kernel, K/V-block outer loop (same review: each CTA owns dK_j, dV_j
//     and needs no inter-CTA synchronisation; dQ is accumulated across CTAs
//     by reduce-adds, here TMA tensor reductions into an fp32 buffer).  Per (b, h, 128-key block j), for each 128-query
//     block i that can see block j:
//        S^T  = K_j Q_i^T              (recomputed; sj-techlog "FlashAttention
//        dP^T = V_j dO_i^T              원 논문 해부", backward section)
//        P^T  = exp(tau S^T - lse_i)   (FlashAttention-2 review, "개선 2")
//        dS^T = P^T o (dP^T - D_i)     (review, "Backward Pass": softmax grad)
//        dQ_i += dS_ij K_j   (fp32 reduce-adds into dq_accum)
//        dV_j += P^T dO_i,   dK_j += dS^T Q_i
//     and finally dK_j *= tau (S = tau Q K^T);
//  3. convert: dQ = tau * dq_accum, rounded to the 16-bit type.
//
// GB300 mapping of the main kernel: see the comment above BwdCfg.
#include "attn_common.cuh"

namespace attn {

// ============================================================================
// 3. dQ convert
// ============================================================================
template <bool BF16>
__global__ void __launch_bounds__(256) attn_dq_convert_kernel(const DqConvertArgs a) {
    const long long n8 = a.elems / 8;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += stride) {
        const float4 x = reinterpret_cast<const float4*>(a.dq_accum)[2 * i];
        const float4 y = reinterpret_cast<const float4*>(a.dq_accum)[2 * i + 1];
        uint4 r;
        r.x = pack2<BF16>(x.x * a.scale, x.y * a.scale);
        r.y = pack2<BF16>(x.z * a.scale, x.w * a.scale);
        r.z = pack2<BF16>(y.x * a.scale, y.y * a.scale);
        r.w = pack2<BF16>(y.z * a.scale, y.w * a.scale);
        reinterpret_cast<uint4*>(a.dq)[i] = r;
    }
}

// ============================================================================
// 1. preprocess: exact D_i = sum_j P_ij dP_ij, and dq_accum := 0
// ============================================================================
// D is the definition of the softmax-gradient row term (FlashAttention-2
// review, "Backward Pass": D_i = sum_j P_ij dP_ij = (P_i o dP_i)^T 1).  The
// review's shortcut rowsum(dO o O) (computed by the preprocess kernel) uses O
// after its rounding to 16 bits; on rows whose softmax is close to one-hot the
// factor dP_ij - D_i of dS cancels and that rounding dominates dQ.  This pass
// recomputes P from lse in fp32 and dP = dO V^T on the tensor cores and sums
// their product per row, so dS = P (dP - D) below uses the same fp32 P and a
// matching D.
//
// One CTA = one (b, h) and 128 query rows; K/V blocks stream through a TMA
// ring; S and dP of a block land in one of two TMEM buffers so the MMAs of
// block j+1 run while the compute warpgroups reduce block j.  Warpgroup c
// (warps 4+4c .. 7+4c) handles key columns [64c, 64c+64) of each block.
template <int D>
struct DsumCfg {
    static constexpr int STAGES = (D == 128) ? 2 : 4;
    static constexpr int KBOX = D / kBoxCols;
    static constexpr int TILE_BYTES = kTile * D * 2;
    static constexpr int Q_OFF = 0;
    static constexpr int DO_OFF = Q_OFF + TILE_BYTES;
    static constexpr int K_OFF = DO_OFF + TILE_BYTES;
    static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
    static constexpr int RED_OFF = V_OFF + STAGES * TILE_BYTES;   // 128 floats
    static constexpr int BAR_OFF = RED_OFF + kTile * 4;
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + STAGES;
    static constexpr int B_KVEMPTY = B_VFULL + STAGES;
    static constexpr int B_SDP = B_KVEMPTY + STAGES;       // [2]
    static constexpr int B_FREE = B_SDP + 2;               // [2] buffer consumed
    static constexpr int B_RED = B_FREE + 2;               // warpgroup 1 partial sums ready
    static constexpr int B_DRAIN = B_RED + 1;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
    static constexpr int THREADS = 384;
    static constexpr uint32_t TMEM_COLS = 512;
    __device__ static constexpr uint32_t s_col(int b) { return 256u * b; }
    __device__ static constexpr uint32_t dp_col(int b) { return 256u * b + 128u; }
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(384, 1)
attn_bwd_dsum_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const DsumArgs args) {
    using C = DsumCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
    float* red = reinterpret_cast<float*>(smem + C::RED_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = args.N;
    const int nblk = (N + kTile - 1) / kTile;
    const int bh = blockIdx.x;                                      // (batch, query head)
    if (grid_block() >= nblk) return;                               // padding CTA
    const int bkv = kv_head(bh, args.H, args.Hkv);                  // its K / V head
    const int qi = nblk - 1 - grid_block();                         // heavy query blocks first
    const int nkv = CAUSAL ? min(nblk, qi + 1) : nblk;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::B_SDP + b), 1);
            mbar_init(bar(C::B_FREE + b), 256);
        }
        mbar_init(bar(C::B_RED), 128);
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = (*reinterpret_cast<volatile int*>(args.status) != 0) ? 1 : 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, args.status, args.wait_polls};
    const bool skip = *abort_flag != 0;

    if (!skip && warp >= 2) {
        // dq_accum := 0 for this CTA's 128 rows (a contiguous 128 x d fp32 block),
        // coalesced, by the warps that are otherwise idle until the first MMA
        const int rows = min(kTile, N - qi * kTile);
        float4* z = reinterpret_cast<float4*>(args.dq_accum +
                                              (static_cast<size_t>(bh) * N + qi * kTile) * D);
        const int n4 = rows * D / 4;
        for (int e = threadIdx.x - 64; e < n4; e += C::THREADS - 64) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    if (skip) {
    } else if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::TILE_BYTES);
            for (int b = 0; b < C::KBOX; ++b) {
                tma_load_3d(sbase + C::Q_OFF + b * kBoxBytes, &tm_q, bar(C::B_QFULL), b * kBoxCols,
                            qi * kTile, bh, pol_q);
                tma_load_3d(sbase + C::DO_OFF + b * kBoxBytes, &tm_do, bar(C::B_QFULL),
                            b * kBoxCols, qi * kTile, bh, pol_q);
            }
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < nkv; ++j) {
                const int s = j % C::STAGES;
                if (j >= C::STAGES) {
                    ok = wait_bar(wc, bar(C::B_KVEMPTY + s), ((j / C::STAGES) - 1) & 1);
                    if (!ok) break;
                }
                mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE_BYTES);
                for (int b = 0; b < C::KBOX; ++b)
                    tma_load_3d(sbase + C::K_OFF + s * C::TILE_BYTES + b * kBoxBytes, &tm_k,
                                bar(C::B_KFULL + s), b * kBoxCols, j * kTile, bkv, pol_kv);
                mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE_BYTES);
                for (int b = 0; b < C::KBOX; ++b)
                    tma_load_3d(sbase + C::V_OFF + s * C::TILE_BYTES + b * kBoxBytes, &tm_v,
                                bar(C::B_VFULL + s), b * kBoxCols, j * kTile, bkv, pol_kv);
                issued = j + 1;
            }
            if (!ok) {
                drain_wait(bar(C::B_QFULL), 0);
                for (int j = max(0, issued - C::STAGES); j < issued; ++j) {
                    drain_wait(bar(C::B_KFULL + j % C::STAGES), (j / C::STAGES) & 1);
                    drain_wait(bar(C::B_VFULL + j % C::STAGES), (j / C::STAGES) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t fmt = BF16 ? 1u : 0u;
            constexpr uint32_t id = idesc_f16(128, 128, fmt, 0, 0);  // Q K^T and dO V^T
            bool ok = wait_bar(wc, bar(C::B_QFULL), 0);
            for (int j = 0; ok && j < nkv; ++j) {
                const int s = j % C::STAGES;
                const int b = j & 1;
                if (!(ok = wait_bar(wc, bar(C::B_KFULL + s), (j / C::STAGES) & 1))) break;
                if (j >= 2 && !(ok = wait_bar(wc, bar(C::B_FREE + b), ((j >> 1) - 1) & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_ss(tmem + C::s_col(b),
                           smem_desc(sbase + C::Q_OFF + off, 16, 1024, LAYOUT_SW128),
                           smem_desc(sbase + C::K_OFF + s * C::TILE_BYTES + off, 16, 1024, LAYOUT_SW128),
                           id, kk > 0);
                }
                if (!(ok = wait_bar(wc, bar(C::B_VFULL + s), (j / C::STAGES) & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_ss(tmem + C::dp_col(b),
                           smem_desc(sbase + C::DO_OFF + off, 16, 1024, LAYOUT_SW128),
                           smem_desc(sbase + C::V_OFF + s * C::TILE_BYTES + off, 16, 1024, LAYOUT_SW128),
                           id, kk > 0);
                }
                mma_commit(bar(C::B_SDP + b));
                mma_commit(bar(C::B_KVEMPTY + s));
            }
            mma_commit(bar(C::B_DRAIN));
            drain_wait(bar(C::B_DRAIN), 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ row sums
        const int c = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const int row = qi * kTile + r;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const float cs = args.scale_log2;
        const float nl2 = (row < N) ? -args.lse[static_cast<size_t>(bh) * N + row] * kLog2e : 0.f;
        uint64_t acc2 = f2_pack(0.f, 0.f);
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            const int b = j & 1;
            ok = __all_sync(0xffffffffu, wait_bar(wc, bar(C::B_SDP + b), (j >> 1) & 1));
            if (!ok) break;
            tc_fence_after();
            // keys >= limit are masked: the key tail and, on the diagonal block, keys > row
            int limit = N - (j * kTile + 64 * c);
            if (CAUSAL) limit = min(limit, row - (j * kTile + 64 * c) + 1);
            // both loads in flight before one wait
            uint32_t sr[64], dr[64];
            tmem_ld_sync(tmem + lane_off + C::s_col(b) + 64 * c, sr, tmem + lane_off + C::dp_col(b) + 64 * c, dr);
            // the buffer can be refilled as soon as it has been read
            tc_fence_before();
            mbar_arrive(bar(C::B_FREE + b));
            const uint64_t cs2 = f2_pack(cs, cs);
            const uint64_t nl22 = f2_pack(nl2, nl2);
            if (limit >= 64) {
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const uint64_t arg = f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                                cs2, nl22);
                    float a0, a1;
                    f2_unpack(arg, a0, a1);
                    acc2 = f2_fma(f2_pack(ex2_approx(a0), ex2_approx(a1)),
                                  f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), acc2);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const uint64_t arg = f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                                cs2, nl22);
                    float a0, a1;
                    f2_unpack(arg, a0, a1);
                    const float p0 = (e >= limit) ? 0.f : ex2_approx(a0);
                    const float p1 = (e + 1 >= limit) ? 0.f : ex2_approx(a1);
                    acc2 = f2_fma(f2_pack(p0, p1),
                                  f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), acc2);
                }
            }
        }
        float acc0, acc1;
        f2_unpack(acc2, acc0, acc1);
        const float acc = acc0 + acc1;
        if (c == 1) {
            red[r] = acc;
            mbar_arrive(bar(C::B_RED));
        } else if (ok) {
            ok = __all_sync(0xffffffffu, wait_bar(wc, bar(C::B_RED), 0));
            if (ok && row < N) args.D[static_cast<size_t>(bh) * N + row] = acc + red[r];
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ============================================================================
// 1c. preprocess from the forward's fp32 O: D_i = sum_k dO_ik O_ik, dq_accum := 0
// ============================================================================
// The FlashAttention-2 review's form of D ("Backward Pass" of FlashAttention-2:
// D_i = rowsum(dO_i o O_i)), evaluated with the fp32 copy of O that
// attn_fwd_train writes.  That O is normalised by the sum of the rounded P
// that multiplied V, so its weights sum to exactly 1 and D matches the P the
// backward recomputes even on nearly one-hot rows.  Memory-bound: one pass
// over O (fp32) and dO, plus zeroing dq_accum.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_o32_kernel(const PreO32Args a) {
    constexpr int TPR = D / 8;  // threads per row, 8 elements each
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const int sub = threadIdx.x % TPR;
    const long long rows_per_sweep = nthreads / TPR;
    const long long sweeps = (a.rows + rows_per_sweep - 1) / rows_per_sweep;
    // every thread runs the same number of sweeps, so the row-group shuffles
    // below always see all 32 lanes of the warp
    for (long long sw = 0; sw < sweeps; ++sw) {
        const long long row = sw * rows_per_sweep + tid / TPR;
        const bool valid = row < a.rows;
        float acc = 0.f;
        if (valid) {
            const float4* o4 = reinterpret_cast<const float4*>(a.o32 + row * D + sub * 8);
            const float4 x0 = o4[0], x1 = o4[1];
            const uint4 d4 = reinterpret_cast<const uint4*>(a.dO)[row * TPR + sub];
            const uint16_t* dh = reinterpret_cast<const uint16_t*>(&d4);
            const float ov[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(ov[e], to_f32<BF16>(dh[e]), acc);
            float4* z = reinterpret_cast<float4*>(a.dq_accum + row * D + sub * 8);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
        if (valid && sub == 0) a.D[row] = acc;
    }
}

// ============================================================================
// 2. main backward kernel
// ============================================================================
// One CTA = one (b, h) and one 128-key block j; it loops over the 128-query
// blocks i that can see block j and keeps dV_j, dK_j in TMEM.  Per block i:
//
//   MMA:   S^T = K Q_i^T, dP^T = V dO_i^T                     (N = 128)
//   WG0/1: P^T = exp2(S^T tau log2e - lse2) for query columns [64c, 64c+64),
//          back into TMEM as 16-bit pairs over the first half of the same
//          columns; later dS^T = P^T (dP^T - D), into TMEM over the first half
//          of the dP^T columns and into shared memory
//   MMA:   dV += P^T dO_i as soon as P^T is in, dK += dS^T Q_i (A from TMEM),
//          dQ = dS K_j
//   WG0/1: dQ rows read out of TMEM, staged in shared memory over the Q_i /
//          dO_i tiles (no longer read by then); warp 2 adds them to dq_accum
//          with TMA tensor reduce-adds and hands the stage back to the TMA
//          producer.
//
// Overlap: the tensor core runs S^T_i, dP^T_i, dV_i, dK_i, dQ_i in that order
// with one barrier per product, so the exponentials of block i overlap dP^T_i
// and the dS_i arithmetic overlaps dV_i.  (Issuing S^T_{i+1} before dQ_i
// would make it wait for the next Q tile, whose stage is only freed once the
// dQ of the block before has been reduced.)
//
// TMEM columns: S^T at 0 (P^T of warpgroup c at 64c, 32 packed columns),
// dP^T at 128 (dS^T of warpgroup c at 128 + 64c; then dQ at 128, d columns),
// dV at 256, dK at 256 + d.  Each warpgroup only overwrites columns it has
// read itself.  dP^T_{i+1} waits until dQ_i has been read out.
template <int D>
struct BwdCfg {
    static constexpr int STAGES = (D == 128) ? 2 : 3;       // Q_i / dO_i ring depth
    static constexpr int KBOX = D / kBoxCols;
    static constexpr int TILE_BYTES = kTile * D * 2;        // 128 x D 16-bit tile
    static constexpr int DS_BYTES = kTile * kTile * 2;      // dS^T, 128 keys x 128 queries
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE_BYTES;
    static constexpr int DS_OFF = V_OFF + TILE_BYTES;
    static constexpr int Q_OFF = DS_OFF + DS_BYTES;
    static constexpr int DO_OFF = Q_OFF + STAGES * TILE_BYTES;
    static constexpr int STAT_OFF = DO_OFF + STAGES * TILE_BYTES;   // lse2[S][128], Dv[S][128]
    static constexpr int BAR_OFF = STAT_OFF + STAGES * 2 * kTile * 4;
    static constexpr int B_KVFULL = 0;
    static constexpr int B_QFULL = 1;
    static constexpr int B_DOFULL = B_QFULL + STAGES;
    static constexpr int B_STFULL = B_DOFULL + STAGES;      // stats ready  [S]
    static constexpr int B_STEMPTY = B_STFULL + STAGES;     // stats free   [S]
    static constexpr int B_SFULL = B_STEMPTY + STAGES;      // S^T in TMEM
    static constexpr int B_DPFULL = B_SFULL + 1;            // dP^T in TMEM
    static constexpr int B_PREADY = B_DPFULL + 1;           // P^T written (S^T read)
    static constexpr int B_DS = B_PREADY + 1;               // dS^T written (dP^T read)
    static constexpr int B_DQFULL = B_DS + 1;               // dQ in TMEM
    static constexpr int B_DQEMPTY = B_DQFULL + 1;          // dQ columns read out
    // dQ staged in smem, one barrier per stage: phase k+1 of STAGED[s] needs
    // stage s reloaded, hence released by the reducer after it saw phase k.
    // (With a single barrier the compute warpgroups could stage two blocks
    // while the reducer still finished the one before, and its parity wait
    // would then miss both phases.)
    static constexpr int B_STAGED = B_DQEMPTY + 1;          // [S]
    static constexpr int B_ACC = B_STAGED + STAGES;         // dV, dK final
    static constexpr int B_EPI = B_ACC + 1;                 // [2] dV / dK rows staged (128 each)
    static constexpr int B_DRAIN = B_EPI + 2;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    // The d=128 layout needs (almost) all 227 KB, so it relies on the dynamic
    // shared-memory window starting 1024-byte aligned (checked at run time).
    static constexpr int SLACK = (D == 128) ? 0 : 1024;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + SLACK;
    // block-sparse variant: the key block's list of kept query blocks
    static constexpr int LIST_OFF = MISC_OFF + 16;
    static constexpr int SMEM_SPARSE = LIST_OFF + 2 * kMaxSparseBlocks + SLACK;
    static constexpr int THREADS = 384;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0, P_COL = 0, DP_COL = 128, DS_COL = 128, DQ_COL = 128;
    static constexpr uint32_t DV_COL = 256, DK_COL = 256 + D;
    static constexpr int DQ_BOX_COLS = 32;                  // fp32 columns per reduce box
    static constexpr int DQ_BOX_BYTES = kTile * DQ_BOX_COLS * 4;   // 16 KB
    static_assert(SMEM_SPARSE <= 232448, "shared memory budget");
    static_assert(D * kTile * 4 <= 2 * TILE_BYTES, "dQ staging fits in the Q_i + dO_i tiles");
};

// Staging address of dQ box b (fp32 columns [32b, 32b+32)) of stage s: boxes
// fill the Q_i tile first, then the dO_i tile.
template <int D>
__device__ __forceinline__ uint32_t dq_box_addr(uint32_t sbase, int s, int b) {
    using C = BwdCfg<D>;
    constexpr int per_tile = C::TILE_BYTES / C::DQ_BOX_BYTES;   // 2 (d=128) or 1 (d=64)
    return sbase + (b < per_tile ? C::Q_OFF : C::DO_OFF) + s * C::TILE_BYTES +
           (b % per_tile) * C::DQ_BOX_BYTES;
}

template <int D, bool CAUSAL, bool BF16, bool GENERAL, bool SPARSE, bool DROPOUT>
__global__ void __launch_bounds__(384, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                const __grid_constant__ CUtensorMap tm_dv, const BwdArgs args) {
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    if (pad > static_cast<uint32_t>(C::SLACK)) {
        // the layout does not fit this placement; report instead of faulting
        if (threadIdx.x == 0) atomicExch(args.status, DEV_SMEM_ALIGN);
        return;
    }
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
    float* stats = reinterpret_cast<float*>(smem + C::STAT_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // (batch, K / V head) and key block (causal: small j = most work).  Dense
    // MHA: head groups, x = head within the group, y = key block, z = group
    // (one group of all heads is the plain order).  Otherwise x = (batch, K / V
    // head) and y / z = key block, or, for a packed batch, head-major: x = key
    // block and y / z = (sequence, K / V head), so the key blocks of one
    // sequence and head run together and the fp32 dQ rows they all reduce into
    // stay in L2.
    int bkv, j;
    if constexpr (!GENERAL) {
        bkv = static_cast<int>(blockIdx.z * gridDim.x + blockIdx.x);
        j = blockIdx.y;
    } else {
        bkv = blockIdx.x;
        j = grid_block();
        if (args.splits > 1) bkv /= args.splits;                 // x = (K / V head, split)
        if (args.cu_seqlens != nullptr) {
            j = blockIdx.x;
            bkv = grid_block();
            if (bkv >= args.BHkv) return;                           // padding CTA
        }
    }
    if (j >= args.num_kvblocks) return;                             // padding CTA
    // GENERAL (grouped K / V heads and / or a packed variable-length batch): the
    // query heads of this K / V head's group, one after the other; block it of
    // the loop is query block qblk(it) of query head qhead(it), and dK_j, dV_j
    // accumulate over all of them.  Rows of the sequence start at token tok0.
    // Otherwise (dense, Hkv = H) the one query head of the same index, without
    // the divisions.  TMA head coordinates: kvc for K, V, dK, dV and qhead(it)
    // for Q, dO, dQ; qflat(it) is the (batch, head) index of the lse / D rows.
    // N, tok0: the query rows; Nk, tokk0: the key rows (the same unless a packed
    // batch gives keys of their own lengths), koff = Nk - N: with a causal mask
    // key j is visible to query i iff j <= i + koff.
    int N = args.N, tok0 = 0, kvc = bkv, qc0 = bkv, qf0 = bkv, group = 1, split = 0;
    int Nk = N, tokk0 = 0, koff = 0;
    bool varlen = false;
    if constexpr (GENERAL) {
        const int b = bkv / args.Hkv, kvh = bkv % args.Hkv;
        group = args.H / args.Hkv;
        qf0 = b * args.H + kvh * group;
        if (args.splits > 1) {
            // this CTA's share of the group: query heads [split * group', (split + 1) * group')
            split = static_cast<int>(blockIdx.x) - bkv * args.splits;
            group /= args.splits;
            qf0 += split * group;
        }
        qc0 = qf0;
        if (args.cu_seqlens != nullptr) {
            varlen = true;
            const int s0 = min(max(args.cu_seqlens[b], 0), args.total);
            const int s1 = min(max(args.cu_seqlens[b + 1], s0), args.total);
            tok0 = s0;
            N = min(s1 - s0, args.max_seqlen);
            tokk0 = tok0;
            Nk = N;
            if (args.cu_seqlens_k != nullptr) {
                const int k0 = min(max(args.cu_seqlens_k[b], 0), args.total_k);
                const int k1 = min(max(args.cu_seqlens_k[b + 1], k0), args.total_k);
                tokk0 = k0;
                Nk = min(k1 - k0, args.max_seqlen_k);
                koff = Nk - N;
            }
            kvc = kvh;
            qc0 = kvh * group;
            if (j * kTile >= Nk) return;                            // not a block of this sequence
        }
    }
    const int nq = GENERAL ? (N + kTile - 1) / kTile : args.num_kvblocks;  // query blocks (dense: == key blocks)
    // causal: the first query that sees key j * kTile is j * kTile - koff
    const int i_start = !CAUSAL ? 0 : GENERAL ? max(0, j * kTile - koff) / kTile : j;
    const int n_i = max(0, nq - i_start);        // query blocks per query head
    int n_it = group * n_i;
    // Block-sparse layout (dense, one query head per CTA): the query blocks
    // visited are those whose tile with key block j is kept, in order, listed
    // by warp 3 before the roles start.
    const uint16_t* blist = reinterpret_cast<const uint16_t*>(smem + C::LIST_OFF);
    if (SPARSE && warp == 3) {
        const uint8_t* mcol = args.block_mask + bkv * args.mask_head_stride + j;
        uint16_t* wl = reinterpret_cast<uint16_t*>(smem + C::LIST_OFF);
        int n = 0;
        for (int c0 = i_start; c0 < nq; c0 += 32) {
            const int i = c0 + lane;
            const bool keep = i < nq && mcol[static_cast<long long>(i) * args.mask_cols] != 0;
            const unsigned bal = __ballot_sync(0xffffffffu, keep);
            if (keep) wl[n + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint16_t>(i);
            n += __popc(bal);
        }
        if (lane == 0) *reinterpret_cast<int*>(smem + C::MISC_OFF + 8) = n;
    }
    auto qhead = [&](int it) { return GENERAL ? qc0 + it / n_i : qc0; };
    auto qflat = [&](int it) { return GENERAL ? qf0 + it / n_i : qf0; };
    auto qblk = [&](int it) -> int {
        return SPARSE ? static_cast<int>(blist[it]) : GENERAL ? i_start + it % n_i : i_start + it;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_KVFULL), 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar(C::B_QFULL + s), 1);
            mbar_init(bar(C::B_DOFULL + s), 1);
            mbar_init(bar(C::B_STFULL + s), 32);
            mbar_init(bar(C::B_STEMPTY + s), 256);
        }
        mbar_init(bar(C::B_SFULL), 1);
        mbar_init(bar(C::B_DPFULL), 1);
        mbar_init(bar(C::B_PREADY), 256);
        mbar_init(bar(C::B_DS), 256);
        mbar_init(bar(C::B_DQFULL), 1);
        mbar_init(bar(C::B_DQEMPTY), 256);
        for (int s = 0; s < C::STAGES; ++s) mbar_init(bar(C::B_STAGED + s), 256);
        mbar_init(bar(C::B_ACC), 1);
        mbar_init(bar(C::B_EPI + 0), 128);
        mbar_init(bar(C::B_EPI + 1), 128);
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = (*reinterpret_cast<volatile int*>(args.status) != 0) ? 1 : 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dq);
        tma_prefetch_desc(&tm_dk);
        tma_prefetch_desc(&tm_dv);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, args.status, args.wait_polls};
    bool skip = *abort_flag != 0;
    if constexpr (SPARSE) {
        n_it = *reinterpret_cast<const int*>(smem + C::MISC_OFF + 8);
        if (n_it == 0 && !skip) {
            // no query block keeps a tile with these keys: dK = dV = 0
            const int rows = min(kTile, N - j * kTile);
            const size_t base = (static_cast<size_t>(bkv) * N + static_cast<size_t>(j) * kTile) * D;
            for (int e = threadIdx.x; e < rows * (D / 8); e += C::THREADS) {
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.dk) + base)[e] = make_uint4(0u, 0u, 0u, 0u);
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.dv) + base)[e] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (n_it == 0) skip = true;
    }
    if constexpr (GENERAL) {
        if (varlen && n_it == 0 && !skip) {
            // a packed sequence with keys but no queries: dK = dV = 0 for these keys
            const int rows = min(kTile, Nk - j * kTile);
            for (int e = threadIdx.x; e < rows * (D / 8); e += C::THREADS) {
                const size_t rb = (static_cast<size_t>(tokk0 + j * kTile + e / (D / 8)) * args.Hkv + kvc) * D;
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.dk) + rb)[e % (D / 8)] = make_uint4(0u, 0u, 0u, 0u);
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.dv) + rb)[e % (D / 8)] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (varlen && n_it == 0) skip = true;
    }

    // Register budgets: 384 threads x 168 registers at launch; the role warps
    // (TMA, MMA, dQ reducer, lse/D loader) need few, the two compute
    // warpgroups many: 128 x 120 + 256 x 192 = 384 x 168.
    static_assert(C::THREADS * 168 == 128 * 120 + 256 * 192, "register split");
    if (warp < 4) {
        regs_dec<120>();
        if (!skip) {
            if (warp == 0) {
                // ------------------------------------------------------------ TMA producer
                if (lane == 0) {
                    const uint64_t pol_kv = policy_evict_first();
                    const uint64_t pol_q = policy_evict_last();
                    mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::TILE_BYTES);
                    for (int b = 0; b < C::KBOX; ++b) {
                        tma_load_3d(sbase + C::K_OFF + b * kBoxBytes, &tm_k, bar(C::B_KVFULL), b * kBoxCols,
                                    tokk0 + j * kTile, kvc, pol_kv);
                        tma_load_3d(sbase + C::V_OFF + b * kBoxBytes, &tm_v, bar(C::B_KVFULL), b * kBoxCols,
                                    tokk0 + j * kTile, kvc, pol_kv);
                    }
                    // Only the first STAGES Q / dO tiles: the dQ reducer reloads each
                    // stage itself as soon as its reductions have read it (see there).
                    for (int it = 0; it < min(n_it, C::STAGES); ++it) {
                        const int i = qblk(it);
                        const int bh = qhead(it);
                        mbar_arrive_expect_tx(bar(C::B_QFULL + it), C::TILE_BYTES);
                        for (int b = 0; b < C::KBOX; ++b)
                            tma_load_3d(sbase + C::Q_OFF + it * C::TILE_BYTES + b * kBoxBytes, &tm_q,
                                        bar(C::B_QFULL + it), b * kBoxCols, tok0 + i * kTile, bh, pol_q);
                        mbar_arrive_expect_tx(bar(C::B_DOFULL + it), C::TILE_BYTES);
                        for (int b = 0; b < C::KBOX; ++b)
                            tma_load_3d(sbase + C::DO_OFF + it * C::TILE_BYTES + b * kBoxBytes, &tm_do,
                                        bar(C::B_DOFULL + it), b * kBoxCols, tok0 + i * kTile, bh, pol_q);
                    }
                }
            } else if (warp == 1) {
                // ------------------------------------------------------------ MMA issuer
                if (lane == 0) {
                    constexpr uint32_t fmt = BF16 ? 1u : 0u;
                    constexpr uint32_t id_kk = idesc_f16(128, 128, fmt, 0, 0);  // K x Q^T, V x dO^T
                    constexpr uint32_t id_acc = idesc_f16(128, D, fmt, 0, 1);   // P^T x dO, dS^T x Q
                    constexpr uint32_t id_dq = idesc_f16(128, D, fmt, 1, 1);    // dS x K (both MN-major)
                    // S^T = K Q_i^T into the S columns, committed to SFULL
                    const uint64_t k_kmaj = smem_desc(sbase + C::K_OFF, 16, 1024, LAYOUT_SW128);
                    const uint64_t v_kmaj = smem_desc(sbase + C::V_OFF, 16, 1024, LAYOUT_SW128);
                    const uint64_t k_mn = smem_desc(sbase + C::K_OFF, kBoxBytes, 1024, LAYOUT_SW128);
                    const uint64_t ds_mn = smem_desc(sbase + C::DS_OFF, kBoxBytes, 1024, LAYOUT_SW128);
                    auto issue_s = [&](int it) {
                        const uint64_t q0 = smem_desc(sbase + C::Q_OFF + (it % C::STAGES) * C::TILE_BYTES, 16, 1024,
                                                      LAYOUT_SW128);
        #pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                            mma_ss(tmem + C::S_COL, desc_advance(k_kmaj, off), desc_advance(q0, off), id_kk, kk > 0);
                        }
                        mma_commit(bar(C::B_SFULL));
                    };
                    bool ok = wait_bar(wc, bar(C::B_KVFULL), 0);
                    for (int it = 0; ok && it < n_it; ++it) {
                        const int s = it % C::STAGES;
                        const uint32_t ph = (it / C::STAGES) & 1;
                        const uint32_t q_s = sbase + C::Q_OFF + s * C::TILE_BYTES;
                        const uint32_t do_s = sbase + C::DO_OFF + s * C::TILE_BYTES;
                        // S^T of this block: the previous P^T was consumed by its dV MMA
                        if (!(ok = wait_bar(wc, bar(C::B_QFULL + s), ph))) break;
                        tc_fence_after();
                        issue_s(it);
                        if (!(ok = wait_bar(wc, bar(C::B_DOFULL + s), ph))) break;
                        // dP^T overwrites the previous block's dQ: wait for its readout
                        if (it > 0 && !(ok = wait_bar(wc, bar(C::B_DQEMPTY), (it - 1) & 1))) break;
                        tc_fence_after();
                        // dP^T = V dO^T
                        const uint64_t do_kmaj = smem_desc(do_s, 16, 1024, LAYOUT_SW128);
        #pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                            mma_ss(tmem + C::DP_COL, desc_advance(v_kmaj, off), desc_advance(do_kmaj, off), id_kk, kk > 0);
                        }
                        mma_commit(bar(C::B_DPFULL));
                        // dV += P^T dO   (K = the 128 queries of block i; query step kk
                        // lives with warpgroup kk / 4)
                        if (!(ok = wait_bar(wc, bar(C::B_PREADY), it & 1))) break;
                        tc_fence_after();
                        const uint64_t do_mn = smem_desc(do_s, kBoxBytes, 1024, LAYOUT_SW128);
        #pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ts(tmem + C::DV_COL, tmem + C::P_COL + 64 * (kk >> 2) + 8 * (kk & 3),
                                   desc_advance(do_mn, kk * 2048), id_acc, (it > 0 || kk > 0) ? 1u : 0u);
                        // dK += dS^T Q
                        if (!(ok = wait_bar(wc, bar(C::B_DS), it & 1))) break;
                        tc_fence_after();
                        const uint64_t q_mn = smem_desc(q_s, kBoxBytes, 1024, LAYOUT_SW128);
        #pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ts(tmem + C::DK_COL, tmem + C::DS_COL + 64 * (kk >> 2) + 8 * (kk & 3),
                                   desc_advance(q_mn, kk * 2048), id_acc, (it > 0 || kk > 0) ? 1u : 0u);
                        // dQ_i = dS K_j   (A = dS^T in smem read MN-major, B = K_j MN-major)
        #pragma unroll
                        for (int kk = 0; kk < kTile / 16; ++kk)
                            mma_ss(tmem + C::DQ_COL, desc_advance(ds_mn, kk * 2048), desc_advance(k_mn, kk * 2048),
                                   id_dq, kk > 0);
                        mma_commit(bar(C::B_DQFULL));
                    }
                    if (ok) mma_commit(bar(C::B_ACC));
                    mma_commit(bar(C::B_DRAIN));
                    drain_wait(bar(C::B_DRAIN), 0);
                }
            } else if (warp == 2) {
                // ------------------------------------------------------------ dQ reducer
                // Adds each staged dQ tile to dq_accum with TMA reduce-adds and then
                // reloads the stage for block it + STAGES.  The reload of Q (needed
                // first, by the next S^T) is issued between the reductions of the
                // boxes staged over Q and those staged over dO: the SM's TMA engine
                // works through its queue in order, so the load does not wait
                // behind the second half of the reduction.
                if (lane == 0) {
                    const uint64_t pol_q = policy_evict_last();
                    constexpr int NB = D / C::DQ_BOX_COLS;
                    constexpr int NB_Q = C::TILE_BYTES / C::DQ_BOX_BYTES;   // boxes over Q_i
                    int issued_q = 0, issued_do = 0;   // blocks whose reloads were issued
                    for (int it = 0; it < n_it; ++it) {
                        const int s = it % C::STAGES;
                        const int nxt = it + C::STAGES;  // block that reuses this stage
                        if (!wait_bar(wc, bar(C::B_STAGED + s), (it / C::STAGES) & 1)) break;
                        fence_proxy_async_smem();
        #pragma unroll
                        for (int b = 0; b < NB_Q; ++b)
                            tma_reduce_add_3d(&tm_dq, dq_box_addr<D>(sbase, s, b), b * C::DQ_BOX_COLS,
                                              tok0 + qblk(it) * kTile, qhead(it));
                        bulk_commit_group();
                        bulk_wait_group_read<0>();
                        if (nxt < n_it) {
                            mbar_arrive_expect_tx(bar(C::B_QFULL + s), C::TILE_BYTES);
                            for (int b = 0; b < C::KBOX; ++b)
                                tma_load_3d(sbase + C::Q_OFF + s * C::TILE_BYTES + b * kBoxBytes, &tm_q,
                                            bar(C::B_QFULL + s), b * kBoxCols, tok0 + qblk(nxt) * kTile, qhead(nxt), pol_q);
                            issued_q = nxt + 1;
                        }
        #pragma unroll
                        for (int b = NB_Q; b < NB; ++b)
                            tma_reduce_add_3d(&tm_dq, dq_box_addr<D>(sbase, s, b), b * C::DQ_BOX_COLS,
                                              tok0 + qblk(it) * kTile, qhead(it));
                        bulk_commit_group();
                        bulk_wait_group_read<0>();
                        if (nxt < n_it) {
                            mbar_arrive_expect_tx(bar(C::B_DOFULL + s), C::TILE_BYTES);
                            for (int b = 0; b < C::KBOX; ++b)
                                tma_load_3d(sbase + C::DO_OFF + s * C::TILE_BYTES + b * kBoxBytes, &tm_do,
                                            bar(C::B_DOFULL + s), b * kBoxCols, tok0 + qblk(nxt) * kTile, qhead(nxt), pol_q);
                            issued_do = nxt + 1;
                        }
                    }
                    bulk_wait_group_read<0>();   // shared memory read; the adds complete with the kernel
                    // Every load of this CTA must land before its shared memory goes
                    // away, also when a role gave up early: wait (bounded, ignoring
                    // the abort flag) for the last load issued into each stage and
                    // for K / V.  On the normal path these phases completed long ago.
                    const int total_q = max(issued_q, min(n_it, C::STAGES));
                    const int total_do = max(issued_do, min(n_it, C::STAGES));
                    drain_wait(bar(C::B_KVFULL), 0);
                    for (int it = max(0, total_q - C::STAGES); it < total_q; ++it)
                        drain_wait(bar(C::B_QFULL + it % C::STAGES), (it / C::STAGES) & 1);
                    for (int it = max(0, total_do - C::STAGES); it < total_do; ++it)
                        drain_wait(bar(C::B_DOFULL + it % C::STAGES), (it / C::STAGES) & 1);
                }
            } else if (warp == 3) {
                // ------------------------------------------------------------ lse / D loader
                for (int it = 0; it < n_it; ++it) {
                    // lse is [B*H, N] (varlen: [B*H, max_seqlen]); D is [B*H, N]
                    // (varlen: [total, H], one stride of H between the rows of a head)
                    const float* lse_g = args.lse + static_cast<size_t>(qflat(it)) *
                                                        (varlen ? args.max_seqlen : N);
                    const float* d_g = varlen ? args.D + static_cast<size_t>(tok0) * args.H + qflat(it) % args.H
                                              : args.D + static_cast<size_t>(qflat(it)) * N;
                    const size_t dstr = varlen ? static_cast<size_t>(args.H) : 1;
                    const int s = it % C::STAGES;
                    if (it >= C::STAGES &&
                        !__all_sync(0xffffffffu, wait_bar(wc, bar(C::B_STEMPTY + s), ((it / C::STAGES) - 1) & 1)))
                        break;
                    const int q0 = qblk(it) * kTile;
                    float* l2 = stats + s * 2 * kTile;
                    float* dv = l2 + kTile;
        #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int qi = q0 + lane * 4 + e;
                        const bool valid = qi < N;
                        // P = exp(tau s - lse) = exp2(tau log2e s - lse log2e); rows past N get P = 0
                        l2[lane * 4 + e] = valid ? -lse_g[qi] * kLog2e : -INFINITY;
                        dv[lane * 4 + e] = valid ? -d_g[qi * dstr] : 0.f;
                    }
                    mbar_arrive(bar(C::B_STFULL + s));
                }
            }
        }
    } else {
        regs_inc<192>();
        if (!skip) {
                // ------------------------------------------------------------ compute warpgroups
                const int c = (warp - 4) >> 2;           // query half handled by this warpgroup
                const int wq = warp & 3;
                const int r = wq * 32 + lane;            // TMEM lane: key row (and query row for dQ)
                const int key = j * kTile + r;
                const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
                const float cs = args.scale_log2;
                const uint64_t cs2 = f2_pack(cs, cs);
                const bool key_ok = key < Nk;
                uint8_t* ds_row = smem + C::DS_OFF + c * kBoxBytes + r * 128;
                float pv[64];        // P^T of this key row, query columns [64c, 64c + 64), fp32
                // dropout: keep bits of this key row for query columns [64c + 32 ch, +32)
                uint32_t kbits[2] = {0u, 0u};
                // P^T_i: wait for S^T_i and block i's statistics, write packed P^T to TMEM
                auto compute_p = [&](int it) -> bool {
                    const int s = it % C::STAGES;
                    const int i = qblk(it);
                    const int qbase = i * kTile + 64 * c;
                    if constexpr (DROPOUT) {
                        // Keep bits of this key row for query columns [qbase, qbase + 64),
                        // computed before S^T is waited for: the four generator calls
                        // are independent chains that run while the tensor core works.
                        // One call per lane and 16 query columns: patch (key patch of
                        // the lane's group, query patch), transposed so that word b
                        // holds key column b, then exchanged so that each lane holds
                        // its key's bytes; bit q of kbits[ch] = query column 32 ch + q.
                        const uint32_t kp = static_cast<uint32_t>((j * kTile + wq * 32) >> 2) + (lane >> 2);
                        const uint32_t t4 = args.drop.drop_t * 0x01010101u;
                        uint4 wv[4];
        #pragma unroll
                        for (int cg = 0; cg < 4; ++cg)      // cg = 2 ch + g
                            wv[cg] = philox4x32_10(
                                make_uint4(kp, static_cast<uint32_t>((qbase + 32 * (cg >> 1)) >> 2) + (lane & 3) + 4 * (cg & 1),
                                           static_cast<uint32_t>(bkv), args.drop.offset),
                                args.drop.seed_lo, args.drop.seed_hi);
        #pragma unroll
                        for (int ch = 0; ch < 2; ++ch) {
                            uint32_t bits = 0u;
        #pragma unroll
                            for (int g = 0; g < 2; ++g) {
                                uint32_t rv[4];
                                exchange_patch_words(transpose_bytes(wv[2 * ch + g]), lane, rv);
        #pragma unroll
                                for (int cpp = 0; cpp < 4; ++cpp) {
                                    const uint32_t m4 = __vcmpltu4(rv[cpp], t4) & 0x08040201u;
                                    bits |= ((m4 * 0x01010101u) >> 24) << (16 * g + 4 * cpp);
                                }
                            }
                            kbits[ch] = bits;
                        }
                    }
                    if (!__all_sync(0xffffffffu, wait_bar(wc, bar(C::B_SFULL), it & 1) &&
                                                     wait_bar(wc, bar(C::B_STFULL + s), (it / C::STAGES) & 1)))
                        return false;
                    tc_fence_after();
                    // per query: -lse*log2e (the loader stores it negated)
                    const float4* l2 = reinterpret_cast<const float4*>(stats + s * 2 * kTile + 64 * c);
                    // masking is needed only for keys past Nk and on blocks that cross
                    // the causal boundary (first query + koff before the last key)
                    const bool masked = !key_ok || (CAUSAL && (GENERAL ? i * kTile + koff < j * kTile + kTile - 1 : i == j));
                    uint32_t pp[32];
                    // two chunks of 32 query columns keep 32 S values live at a time
        #pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        // masked columns of this chunk are those below lim (query + koff
                        // precedes the key; all of them past the key tail)
                        const int lim = key_ok ? key - koff - (qbase + 32 * ch) : 32;
                        uint32_t sr[32];
                        tmem_ld_sync(tmem + lane_off + C::S_COL + 64 * c + 32 * ch, sr);
        #pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 nl = l2[8 * ch + e4];      // broadcast loads
                            const uint64_t nl2[2] = {f2_pack(nl.x, nl.y), f2_pack(nl.z, nl.w)};
        #pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int q = 4 * e4 + 2 * u;        // column within the chunk
                                // P = exp2(s tau log2e - lse log2e), two queries per instruction
                                const uint64_t arg = f2_fma(f2_pack(__uint_as_float(sr[q]), __uint_as_float(sr[q + 1])),
                                                            cs2, nl2[u]);
                                float a0, a1;
                                f2_unpack(arg, a0, a1);
                                float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
                                if (masked) {
                                    if (q < lim) p0 = 0.f;
                                    if (q + 1 < lim) p1 = 0.f;
                                }
                                pv[32 * ch + q] = p0;
                                pv[32 * ch + q + 1] = p1;
                                pp[16 * ch + 2 * e4 + u] = pack2<BF16>(p0, p1);
                                if constexpr (DROPOUT) {   // dV takes the kept P only
                                    const uint32_t b2 = (kbits[ch] >> q) & 3u;
                                    pp[16 * ch + 2 * e4 + u] &= ((b2 & 1u) * 0xFFFFu) | ((b2 >> 1) * 0xFFFF0000u);
                                }
                            }
                        }
                    }
                    // over columns [64c, 64c + 32): read above by this thread only
                    tmem_st32(tmem + lane_off + C::P_COL + 64 * c, pp);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bar(C::B_PREADY));
                    return true;
                };
                // dS^T_i = P^T (dP^T - D): TMEM (for dK) and shared memory (for dQ)
                auto compute_ds = [&](int it) -> bool {
                    const int s = it % C::STAGES;
                    if (!__all_sync(0xffffffffu, wait_bar(wc, bar(C::B_DPFULL), it & 1))) return false;
                    tc_fence_after();
                    const float4* dvv = reinterpret_cast<const float4*>(stats + s * 2 * kTile + kTile + 64 * c);
                    uint32_t pd[32];
        #pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t dr[32];
                        tmem_ld_sync(tmem + lane_off + C::DP_COL + 64 * c + 32 * ch, dr);
        #pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 nd = dvv[8 * ch + e4];      // -D, broadcast loads
                            const uint64_t nd2[2] = {f2_pack(nd.x, nd.y), f2_pack(nd.z, nd.w)};
        #pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int q = 4 * e4 + 2 * u;
                                uint64_t dp2 = f2_pack(__uint_as_float(dr[q]), __uint_as_float(dr[q + 1]));
                                if constexpr (DROPOUT) {   // dP = Z o (dO V^T) * 256 / t
                                    const uint32_t b2 = (kbits[ch] >> q) & 3u;
                                    const float w = args.drop.drop_scale;
                                    dp2 = f2_mul(dp2, f2_pack((b2 & 1u) ? w : 0.f, (b2 & 2u) ? w : 0.f));
                                }
                                const uint64_t dsv = f2_mul(f2_pack(pv[32 * ch + q], pv[32 * ch + q + 1]),
                                                            f2_add(dp2, nd2[u]));
                                float d0, d1;
                                f2_unpack(dsv, d0, d1);
                                pd[16 * ch + 2 * e4 + u] = pack2<BF16>(d0, d1);
                            }
                        }
                    }
                    // over dP^T columns [64c, 64c + 32): read above by this thread only
                    tmem_st32(tmem + lane_off + C::DS_COL + 64 * c, pd);
                    // dS^T row -> shared memory, 128-byte swizzle: 16-byte chunk k of row
                    // r sits at chunk position k ^ (r % 8).  dQ of the previous block,
                    // the last reader of this buffer, completed before its readout.
        #pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<uint4*>(ds_row + ((k ^ (r & 7)) * 16)) =
                            make_uint4(pd[4 * k], pd[4 * k + 1], pd[4 * k + 2], pd[4 * k + 3]);
                    tmem_st_wait();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(C::B_DS));
                    mbar_arrive(bar(C::B_STEMPTY + s));
                    return true;
                };
                // dQ_i readout (lane = query row of block i) and staging for the reducer
                auto readout_dq = [&](int it) -> bool {
                    const int s = it % C::STAGES;
                    if (!__all_sync(0xffffffffu, wait_bar(wc, bar(C::B_DQFULL), it & 1))) return false;
                    tc_fence_after();
                    constexpr int NQ = D / 2;                 // dQ columns per warpgroup
                    uint32_t q32[NQ];
                    tmem_ld_sync(tmem + lane_off + C::DQ_COL + NQ * c, q32);
                    tc_fence_before();
                    mbar_arrive(bar(C::B_DQEMPTY));
                    // boxes of 32 fp32 columns, 128-byte swizzle: 16-byte chunk k of row r
                    // at chunk position k ^ (r % 8)
        #pragma unroll
                    for (int h = 0; h < NQ / 32; ++h) {
                        uint8_t* box = smem + (dq_box_addr<D>(sbase, s, c * (NQ / 32) + h) - sbase) + r * 128;
        #pragma unroll
                        for (int k = 0; k < 8; ++k)
                            *reinterpret_cast<uint4*>(box + ((k ^ (r & 7)) * 16)) =
                                make_uint4(q32[32 * h + 4 * k], q32[32 * h + 4 * k + 1],
                                           q32[32 * h + 4 * k + 2], q32[32 * h + 4 * k + 3]);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(bar(C::B_STAGED + s));
                    return true;
                };
                bool ok = true;
                for (int it = 0; ok && it < n_it; ++it)
                    ok = compute_p(it) && compute_ds(it) && readout_dq(it);
                // ------------------------------------------------------------ epilogue: dV (c=0), dK (c=1)
                // At d = 128 the rounded rows are staged in the 128-byte-swizzled box
                // layout over the V (dV) or K (dK) tile, no longer read once every MMA
                // has completed, and written out with TMA tensor stores by the
                // warpgroup's first thread; at d = 64 each thread stores its row.
                if (ok) ok = __all_sync(0xffffffffu, wait_bar(wc, bar(C::B_ACC), 0));
                if (ok) {
                    tc_fence_after();
                    // dV summed the kept P unscaled: apply 256 / t here under dropout
                    const float mul = (c == 0) ? (DROPOUT ? args.drop.drop_scale : 1.0f) : args.scale;
                    const uint32_t col = (c == 0) ? C::DV_COL : C::DK_COL;
                    const int region = (c == 0) ? C::V_OFF : C::K_OFF;
                    uint8_t* stage_row = smem + region + r * 128;
                    // Each thread stores its own key row from registers (rows past the
                    // sequence are not written) for the last, partial key block of a
                    // packed sequence, where a TMA box would also cover the first rows
                    // of the next sequence, and always at d = 64, where these stores
                    // running beside the last dQ reduce-adds beat queueing behind them
                    // in the copy engine (at d = 128 the TMA stores are faster).
                    const bool direct = D == 64 || (varlen && (j + 1) * kTile > Nk);
                    // fp32 output (written, or added to a running sum, row by row)
                    const bool f32out = GENERAL && args.dk32 != nullptr;
                    const size_t krow = static_cast<size_t>(j) * kTile + r;
                    uint16_t* drow = static_cast<uint16_t*>(c == 0 ? args.dv : args.dk) +
                                     (varlen ? (static_cast<size_t>(tokk0) + krow) * args.Hkv + kvc
                                             : static_cast<size_t>(kvc) * N + krow) * D;
        #pragma unroll
                    for (int cc = 0; cc < D; cc += 32) {
                        uint32_t a32[32];
                        tmem_ld_sync(tmem + lane_off + col + cc, a32);
                        if (f32out) {
                            if (key_ok) {
                                float* frow = (c == 0 ? args.dv32 : args.dk32) + split * args.split_stride +
                                              (static_cast<size_t>(kvc) * N + j * kTile + r) * D + cc;
        #pragma unroll
                                for (int v4 = 0; v4 < 8; ++v4) {
                                    float4 o = make_float4(__uint_as_float(a32[4 * v4]) * mul,
                                                           __uint_as_float(a32[4 * v4 + 1]) * mul,
                                                           __uint_as_float(a32[4 * v4 + 2]) * mul,
                                                           __uint_as_float(a32[4 * v4 + 3]) * mul);
                                    if (args.acc32) {
                                        const float4 p = *reinterpret_cast<const float4*>(frow + 4 * v4);
                                        o.x += p.x; o.y += p.y; o.z += p.z; o.w += p.w;
                                    }
                                    *reinterpret_cast<float4*>(frow + 4 * v4) = o;
                                }
                            }
                            continue;
                        }
                        uint32_t pk[16];
        #pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack2<BF16>(__uint_as_float(a32[2 * e]) * mul,
                                                __uint_as_float(a32[2 * e + 1]) * mul);
                        if (direct) {
                            if (key_ok) {
        #pragma unroll
                                for (int v4 = 0; v4 < 4; ++v4)
                                    *reinterpret_cast<uint4*>(drow + cc + 8 * v4) =
                                        make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                            }
                            continue;
                        }
                        uint8_t* box_row = stage_row + (cc / 64) * kBoxBytes;
                        const int ch0 = (cc % 64) / 8;
        #pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            *reinterpret_cast<uint4*>(box_row + (((ch0 + v4) ^ (r & 7)) * 16)) =
                                make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                    if (direct || f32out) ok = false;   // stored; skip the TMA store below
                    if (ok) {
                        fence_proxy_async_smem();
                        mbar_arrive(bar(C::B_EPI + c));
                    }
                    if (ok && wq == 0 && lane == 0 && wait_bar(wc, bar(C::B_EPI + c), 0)) {
                        for (int b = 0; b < D / 64; ++b)
                            tma_store_3d(c == 0 ? &tm_dv : &tm_dk, sbase + region + b * kBoxBytes, 64 * b,
                                         tokk0 + j * kTile, kvc);
                        bulk_commit_group();
                        bulk_wait_group_read<0>();   // shared memory read; writes complete with the kernel
                    }
                }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ============================================================================
// launchers
// ============================================================================

cudaError_t launch_bwd_preprocess_o32(const PreO32Args& a, bool bf16, cudaStream_t stream) {
    const long long rows_per_block = 256 / (a.d / 8);
    long long blocks = (a.rows + rows_per_block - 1) / rows_per_block;
    const long long cap = static_cast<long long>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (a.d == 64) {
        if (bf16) attn_bwd_preprocess_o32_kernel<true, 64><<<blocks, 256, 0, stream>>>(a);
        else attn_bwd_preprocess_o32_kernel<false, 64><<<blocks, 256, 0, stream>>>(a);
    } else if (a.d == 128) {
        if (bf16) attn_bwd_preprocess_o32_kernel<true, 128><<<blocks, 256, 0, stream>>>(a);
        else attn_bwd_preprocess_o32_kernel<false, 128><<<blocks, 256, 0, stream>>>(a);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_dq_convert(const DqConvertArgs& a, bool bf16, cudaStream_t stream) {
    long long blocks = (a.elems / 8 + 255) / 256;
    const long long cap = static_cast<long long>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (bf16) attn_dq_convert_kernel<true><<<blocks, 256, 0, stream>>>(a);
    else attn_dq_convert_kernel<false><<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int D, bool CAUSAL, bool BF16, bool GENERAL, bool SPARSE = false, bool DROPOUT = false>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                                const CUtensorMap& tdv, const BwdArgs& a, int BH, cudaStream_t stream) {
    using C = BwdCfg<D>;
    auto kern = attn_bwd_kernel<D, CAUSAL, BF16, GENERAL, SPARSE, DROPOUT>;
    constexpr int smem = SPARSE ? C::SMEM_SPARSE : C::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // packed batch: x = key block, y / z = (sequence, K / V head)
    const dim3 grid = !GENERAL ? group_grid(a.num_kvblocks, BH, a.head_group > 0 ? a.head_group : BH)
                      : a.cu_seqlens != nullptr ? head_major_grid(a.num_kvblocks, BH)
                                                : lpt_grid(a.num_kvblocks, BH * (a.splits > 1 ? a.splits : 1));
    kern<<<grid, C::THREADS, smem, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, a);
    return cudaGetLastError();
}

template <int D, bool CAUSAL, bool BF16>
static cudaError_t launch_pre_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const DsumArgs& a, int BH,
                                 cudaStream_t stream) {
    using C = DsumCfg<D>;
    auto kern = attn_bwd_dsum_kernel<D, CAUSAL, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const dim3 grid = lpt_grid((a.N + kTile - 1) / kTile, BH);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const DsumArgs& a, int BH, int d, bool causal,
                            bool bf16, cudaStream_t stream) {
#define ATTN_PRE_CASE(D_, C_, B_) \
    if (d == D_ && causal == C_ && bf16 == B_) return launch_pre_t<D_, C_, B_>(tq, tk, tv, tdo, a, BH, stream);
    ATTN_PRE_CASE(64, false, true)
    ATTN_PRE_CASE(64, true, true)
    ATTN_PRE_CASE(128, false, true)
    ATTN_PRE_CASE(128, true, true)
    ATTN_PRE_CASE(64, false, false)
    ATTN_PRE_CASE(64, true, false)
    ATTN_PRE_CASE(128, false, false)
    ATTN_PRE_CASE(128, true, false)
#undef ATTN_PRE_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const BwdArgs& a, int BH, int d, bool causal,
                       bool bf16, cudaStream_t stream) {
    // the dense MHA kernel's head-group grid holds at most 65,535 key blocks
    const bool general = a.Hkv != a.H || a.cu_seqlens != nullptr || a.num_kvblocks > kMaxGridY ||
                         a.dk32 != nullptr || a.splits > 1;
    if (a.splits > 1 && (a.cu_seqlens != nullptr || a.dk32 == nullptr)) return cudaErrorInvalidValue;
    const bool sparse = a.block_mask != nullptr;   // dense layout, Hkv = H only
    const bool dropout = a.drop.drop_t > 0 && a.drop.drop_t < 256;   // dense layout, Hkv = H only
    if ((sparse || dropout) && general) return cudaErrorInvalidValue;
    if (sparse && dropout) return cudaErrorInvalidValue;
#define ATTN_BWD_CASE(D_, C_, B_)                                                              \
    if (d == D_ && causal == C_ && bf16 == B_)                                                 \
        return dropout ? launch_bwd_t<D_, C_, B_, false, false, true>(tq, tk, tv, tdo, tdq, tdk, tdv, a, BH, stream) \
             : sparse ? launch_bwd_t<D_, C_, B_, false, true>(tq, tk, tv, tdo, tdq, tdk, tdv, a, BH, stream) \
             : general ? launch_bwd_t<D_, C_, B_, true>(tq, tk, tv, tdo, tdq, tdk, tdv, a, BH, stream) \
                       : launch_bwd_t<D_, C_, B_, false>(tq, tk, tv, tdo, tdq, tdk, tdv, a, BH, stream);
    ATTN_BWD_CASE(64, false, true)
    ATTN_BWD_CASE(64, true, true)
    ATTN_BWD_CASE(128, false, true)
    ATTN_BWD_CASE(128, true, true)
    ATTN_BWD_CASE(64, false, false)
    ATTN_BWD_CASE(64, true, false)
    ATTN_BWD_CASE(128, false, false)
    ATTN_BWD_CASE(128, true, false)
#undef ATTN_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace attn
