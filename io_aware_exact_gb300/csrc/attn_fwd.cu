// attn_fwd.cu - exact attention forward for sm_103a (TMA + tcgen05 + TMEM).
//
// Computes, per (batch, head), O = softmax(tau Q K^T [+ causal mask]) V and
// lse_i = ln sum_j exp(tau q_i.k_j) without writing any N x N matrix.
//
// Algorithm: the FlashAttention-2 forward (wonbeomjang.kr FlashAttention-2
// review, "결과: FlashAttention-2 Forward 알고리즘"): Q-block outer loop
// parallel over CTAs, K/V-block inner loop, running row max m and normaliser l,
// unnormalised accumulator rescaled by exp(m_old - m_new), one division by l at
// the end ("개선 1"), and the logsumexp L = m + log l stored for the backward
// ("개선 2").  The merge rule is the one of sj-techlog "FlashAttention 원 논문
// 해부", section "두 tile을 한 row로 합치는 식".  Fully masked causal tiles are
// skipped ("Causal Masking 최적화" in the FlashAttention-2 review).
//
// GB300 mapping (our design, not the pages'):
//  * one CTA = one (b, h) and 256 query rows, as two 128-row tiles that
//    ping-pong on the tensor core: while the softmax warpgroup of one tile
//    works, the MMAs of the other tile run;
//  * warp 0 issues TMA loads (Q once, K/V through a multi-stage ring), warp 1
//    issues tcgen05.mma from one thread, warp 2 owns the TMEM allocation,
//    warps 4-7 and 8-11 are the softmax warpgroups of tile 0 and tile 1 (one
//    thread per query row, since TMEM lane = row);
//  * S = Q K^T lands in TMEM (fp32, 128 columns per tile); the softmax writes
//    P as packed 16-bit pairs over the first 64 columns of the same region and
//    the PV MMA reads P straight from TMEM; O accumulates in TMEM;
//  * exponentials are exp2 with tau*log2(e) folded into one FMA; the running
//    reference max is only moved when the row max grows by more than 2^8
//    (exact: O and l always share the same reference, so the final O/l and
//    lse are unchanged; it only bounds P by 256);
//  * every wait is bounded; a timeout sets the device status word and the CTA
//    drains its in-flight copies and MMAs, frees TMEM and exits.
#include "attn_common.cuh"

namespace attn {

template <int D>
struct FwdCfg {
    static constexpr int TILES = 2;                       // 128-row Q tiles per CTA
    static constexpr int STAGES = (D == 128) ? 2 : 4;     // K/V ring depth
    static constexpr int TILE_BYTES = kTile * D * 2;      // one 128 x D tile
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILES * TILE_BYTES;
    static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
    static constexpr int BAR_OFF = V_OFF + STAGES * TILE_BYTES;
    // barrier slots
    static constexpr int B_QFULL = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_VFULL = B_KFULL + STAGES;
    // A K stage frees when the S MMAs of its block complete, a V stage when its
    // PV MMAs do, one block later: separate barriers let the producer refill
    // the K stage a whole block earlier than one shared barrier would.
    static constexpr int B_KEMPTY = B_VFULL + STAGES;
    static constexpr int B_VEMPTY = B_KEMPTY + STAGES;
    static constexpr int B_SFULL = B_VEMPTY + STAGES;     // [2]
    static constexpr int B_PFULL = B_SFULL + 2;           // [2]
    static constexpr int B_OFULL = B_PFULL + 2;           // [2]
    static constexpr int B_EPI_STAGED = B_OFULL + 2;      // [2] 16-bit O staged (128 arrivals)
    static constexpr int B_DRAIN = B_EPI_STAGED + 2;
    static constexpr int NUM_BARS = B_DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + runtime alignment slack
    // block-sparse variant: the CTA's list of kept key blocks after the misc words
    static constexpr int LIST_OFF = MISC_OFF + 16;
    static constexpr int SMEM_SPARSE = LIST_OFF + 2 * kMaxSparseBlocks + 1024;
    static constexpr int THREADS = 384;
    static constexpr uint32_t TMEM_COLS = 512;
    // TMEM columns: S/P of tile t at 128*t, O of tile t at 256 + D*t.
    __device__ static constexpr uint32_t s_col(int t) { return 128u * t; }
    __device__ static constexpr uint32_t o_col(int t) { return 256u + D * t; }
    static_assert(SMEM_SPARSE <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL, bool BF16, bool TRAIN, bool VARLEN, bool SPARSE, bool DROPOUT>
__global__ void __launch_bounds__(384, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const __grid_constant__ CUtensorMap tm_o32, const FwdArgs args) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Dense: head groups, x = head within the group, y = block rank, z =
    // group (one group of all heads is the plain order).  Packed batch:
    // head-major, x = block rank, y / z = (sequence, query head).  Either way
    // the CTAs that re-read the same K / V run close together.
    const int bh = VARLEN ? grid_block() : static_cast<int>(blockIdx.z * gridDim.x + blockIdx.x);
    const int rank = VARLEN ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.y);
    if (rank >= args.num_qblocks || (VARLEN && bh >= args.BH)) return;   // padding CTA
    int qb = args.num_qblocks - 1 - rank;                          // heavy blocks first
    // TMA coordinates: the rows of this sequence start at tok0, the head
    // coordinate is hq for Q / O and hk for K / V.  Dense [B,H,N,d]: tok0 = 0
    // and the head coordinate is the (batch, head) index.  Packed variable
    // length [total, H, d]: tok0 is the sequence's first token, N its length.
    int tok0 = 0, N = args.N, hq = bh;
    int hk = kv_head(bh, args.H, args.Hkv);                        // its K / V head
    // Keys: Nk rows from token tokk0; causal offset koff = Nk - N (key j is
    // visible to query i iff j <= i + koff).  Equal to the queries' unless a
    // packed batch gives keys of their own lengths.
    int tokk0 = 0, Nk = N, koff = 0;
    if constexpr (VARLEN) {
        const int b = bh / args.H, h = bh % args.H;
        const int s0 = min(max(args.cu_seqlens[b], 0), args.total);
        const int s1 = min(max(args.cu_seqlens[b + 1], s0), args.total);
        tok0 = s0;
        N = min(s1 - s0, args.max_seqlen);
        hq = h;
        hk = h / (args.H / args.Hkv);
        qb = (N + C::TILES * kTile - 1) / (C::TILES * kTile) - 1 - rank;
        if (qb < 0) return;                                        // past this sequence
        tokk0 = tok0;
        Nk = N;
        if (args.cu_seqlens_k != nullptr) {
            const int k0 = min(max(args.cu_seqlens_k[b], 0), args.total_k);
            const int k1 = min(max(args.cu_seqlens_k[b + 1], k0), args.total_k);
            tokk0 = k0;
            Nk = min(k1 - k0, args.max_seqlen_k);
            koff = Nk - N;
        }
    }
    const int q0 = qb * (C::TILES * kTile);
    const int nkv_all = (Nk + kTile - 1) / kTile;
    int nkv[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int r0 = q0 + kTile * t;
        // causal: the tile's last row sees keys up to that row + koff
        const int last_key = min(r0 + kTile, N) - 1 + koff;
        nkv[t] = (r0 >= N) ? 0 : (CAUSAL ? (last_key < 0 ? 0 : min(nkv_all, last_key / kTile + 1)) : nkv_all);
    }
    int n_iter = max(nkv[0], nkv[1]);

    // Block-sparse layout: the key blocks the CTA visits are those that either
    // of its two query tiles keeps (within its causal range), in order.  Entry
    // = key block | 1 << 14 if tile 0 keeps it | 1 << 15 if tile 1 does; a tile
    // that drops a listed block gives it P = 0.  Built by warp 3 before the
    // roles start.
    const uint16_t* blist = reinterpret_cast<const uint16_t*>(smem + C::LIST_OFF);
    if (SPARSE && warp == 3) {
        const uint8_t* mrow0 = args.block_mask + bh * args.mask_head_stride +
                               static_cast<long long>(q0 / kTile) * args.mask_cols;
        uint16_t* wl = reinterpret_cast<uint16_t*>(smem + C::LIST_OFF);
        int n = 0;
        for (int c0 = 0; c0 < n_iter; c0 += 32) {
            const int kb = c0 + lane;
            const bool a0 = kb < nkv[0] && mrow0[kb] != 0;
            const bool a1 = kb < nkv[1] && mrow0[args.mask_cols + kb] != 0;
            const unsigned bal = __ballot_sync(0xffffffffu, a0 || a1);
            if (a0 || a1)
                wl[n + __popc(bal & ((1u << lane) - 1u))] =
                    static_cast<uint16_t>(kb | (a0 ? 1 << 14 : 0) | (a1 ? 1 << 15 : 0));
            n += __popc(bal);
        }
        if (lane == 0) *reinterpret_cast<int*>(smem + C::MISC_OFF + 8) = n;
    }
    auto kblk = [&](int j) -> int { return SPARSE ? (blist[j] & 0x3FFF) : j; };

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
            mbar_init(bar(C::B_VEMPTY + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::B_SFULL + t), 1);
            mbar_init(bar(C::B_PFULL + t), 128);
            mbar_init(bar(C::B_OFULL + t), 1);
            mbar_init(bar(C::B_EPI_STAGED + t), 128);
        }
        mbar_init(bar(C::B_DRAIN), 1);
        // A failure recorded earlier on this device turns later CTAs into
        // no-ops until the host reads and clears the status word.
        *abort_flag = (*reinterpret_cast<volatile int*>(args.status) != 0) ? 1 : 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
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
        n_iter = *reinterpret_cast<const int*>(smem + C::MISC_OFF + 8);
#pragma unroll
        for (int t = 0; t < 2; ++t) nkv[t] = nkv[t] > 0 ? n_iter : 0;
        if (n_iter == 0 && !skip) {
            // every tile of these rows is dropped: empty softmax, O = 0, lse = -inf
            const int rows = min(C::TILES * kTile, N - q0);
            const size_t base = (static_cast<size_t>(bh) * N + q0) * D;
            for (int e = threadIdx.x; e < rows * (D / 8); e += C::THREADS)
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + base)[e] = make_uint4(0u, 0u, 0u, 0u);
            if (TRAIN)
                for (int e = threadIdx.x; e < rows * (D / 4); e += C::THREADS)
                    reinterpret_cast<float4*>(args.o32 + base)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int e = threadIdx.x; e < rows; e += C::THREADS)
                args.lse[static_cast<size_t>(bh) * N + q0 + e] = -INFINITY;
        }
        if (n_iter == 0) skip = true;
    }
    if constexpr (VARLEN) {
        if (n_iter == 0 && !skip) {
            // no row of this CTA sees a key (keys of length 0, or a causal offset
            // that leaves every row before the first key): O = 0, lse = -inf
            const int rows = min(C::TILES * kTile, N - q0);
            for (int e = threadIdx.x; e < rows * (D / 8); e += C::THREADS) {
                const size_t rb = (static_cast<size_t>(tok0 + q0 + e / (D / 8)) * args.H + hq) * D;
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + rb)[e % (D / 8)] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (TRAIN)
                for (int e = threadIdx.x; e < rows * (D / 4); e += C::THREADS) {
                    const size_t rb = (static_cast<size_t>(tok0 + q0 + e / (D / 4)) * args.H + hq) * D;
                    reinterpret_cast<float4*>(args.o32 + rb)[e % (D / 4)] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            for (int e = threadIdx.x; e < rows; e += C::THREADS)
                args.lse[static_cast<size_t>(bh) * args.max_seqlen + q0 + e] = -INFINITY;
        }
        if (n_iter == 0) skip = true;
    }

    if (warp < 4) {
        if (skip) {
            // nothing issued, nothing to drain
        } else if (warp == 0) {
            // ------------------------------------------------------------ TMA producer
            if (lane == 0) {
                const uint64_t pol_q = policy_evict_first();
                const uint64_t pol_kv = policy_evict_last();
                const int ntiles = (nkv[1] > 0) ? 2 : 1;
                mbar_arrive_expect_tx(bar(C::B_QFULL), ntiles * C::TILE_BYTES);
                for (int t = 0; t < ntiles; ++t)
                    tma_load_4d(sbase + C::Q_OFF + t * C::TILE_BYTES, &tm_q, bar(C::B_QFULL), 0,
                                tok0 + q0 + kTile * t, 0, hq, pol_q);
                // K_j and V_j, one copy each; K_j waits for its stage's K to be
                // free, V_j for its V (the K stage frees first)
                int issued_k = 0, issued_v = 0;
                bool ok = true;
                for (int j = 0; j < n_iter; ++j) {
                    const int s = j % C::STAGES;
                    const uint32_t ph = ((j / C::STAGES) - 1) & 1;
                    if (j >= C::STAGES && !(ok = wait_bar(wc, bar(C::B_KEMPTY + s), ph))) break;
                    mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE_BYTES);
                    tma_load_4d(sbase + C::K_OFF + s * C::TILE_BYTES, &tm_k, bar(C::B_KFULL + s), 0,
                                tokk0 + kblk(j) * kTile, 0, hk, pol_kv);
                    issued_k = j + 1;
                    if (j >= C::STAGES && !(ok = wait_bar(wc, bar(C::B_VEMPTY + s), ph))) break;
                    mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE_BYTES);
                    tma_load_4d(sbase + C::V_OFF + s * C::TILE_BYTES, &tm_v, bar(C::B_VFULL + s), 0,
                                tokk0 + kblk(j) * kTile, 0, hk, pol_kv);
                    issued_v = j + 1;
                }
                if (!ok) {
                    // let copies already in flight land before the CTA's smem goes away
                    drain_wait(bar(C::B_QFULL), 0);
                    for (int j = max(0, issued_k - C::STAGES); j < issued_k; ++j)
                        drain_wait(bar(C::B_KFULL + j % C::STAGES), (j / C::STAGES) & 1);
                    for (int j = max(0, issued_v - C::STAGES); j < issued_v; ++j)
                        drain_wait(bar(C::B_VFULL + j % C::STAGES), (j / C::STAGES) & 1);
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            if (lane == 0) {
                constexpr uint32_t fmt = BF16 ? 1u : 0u;
                constexpr uint32_t idesc_s = idesc_f16(128, 128, fmt, 0, 0);  // Q (K-major) x K (K-major)
                constexpr uint32_t idesc_o = idesc_f16(128, D, fmt, 0, 1);    // P (TMEM) x V (MN-major)
                auto issue_s = [&](int t, int s) {
                    const uint64_t a0 = smem_desc(sbase + C::Q_OFF + t * C::TILE_BYTES, 16, 1024, LAYOUT_SW128);
                    const uint64_t b0 = smem_desc(sbase + C::K_OFF + s * C::TILE_BYTES, 16, 1024, LAYOUT_SW128);
    #pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                        mma_ss(tmem + C::s_col(t), desc_advance(a0, off), desc_advance(b0, off), idesc_s,
                               kk > 0 ? 1u : 0u);
                    }
                };
                auto issue_pv = [&](int t, int s, bool acc) {
                    const uint64_t b0 = smem_desc(sbase + C::V_OFF + s * C::TILE_BYTES, kBoxBytes, 1024, LAYOUT_SW128);
    #pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ts(tmem + C::o_col(t), tmem + C::s_col(t) + kk * 8, desc_advance(b0, kk * 2048), idesc_o,
                               (acc || kk > 0) ? 1u : 0u);
                };
                bool ok = wait_bar(wc, bar(C::B_QFULL), 0) && wait_bar(wc, bar(C::B_KFULL + 0), 0);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < 2; ++t)
                        if (nkv[t] > 0) {
                            issue_s(t, 0);
                            mma_commit(bar(C::B_SFULL + t));
                        }
                    mma_commit(bar(C::B_KEMPTY + 0));   // K_0 read by both S MMAs
                }
                for (int j = 0; ok && j < n_iter; ++j) {
                    const int s = j % C::STAGES;
                    if (!(ok = wait_bar(wc, bar(C::B_VFULL + s), (j / C::STAGES) & 1))) break;
                    bool next_k_ready = false;
                    const int t_last = (j < nkv[1]) ? 1 : 0;   // last tile that reads V_j
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= nkv[t]) continue;
                        if (!(ok = wait_bar(wc, bar(C::B_PFULL + t), j & 1))) break;
                        tc_fence_after();
                        issue_pv(t, s, j > 0);
                        if (t == t_last) mma_commit(bar(C::B_VEMPTY + s));   // V_j read by its PV MMAs
                        if (j + 1 < nkv[t]) {
                            if (!next_k_ready) {
                                const int s1 = (j + 1) % C::STAGES;
                                if (!(ok = wait_bar(wc, bar(C::B_KFULL + s1), ((j + 1) / C::STAGES) & 1)))
                                    break;
                                tc_fence_after();
                                next_k_ready = true;
                            }
                            issue_s(t, (j + 1) % C::STAGES);
                            mma_commit(bar(C::B_SFULL + t));
                        } else {
                            mma_commit(bar(C::B_OFULL + t));
                        }
                    }
                    // K_{j+1} read by the S MMAs just issued
                    if (next_k_ready) mma_commit(bar(C::B_KEMPTY + (j + 1) % C::STAGES));
                }
                // make sure no MMA is still reading smem / writing TMEM at teardown
                mma_commit(bar(C::B_DRAIN));
                drain_wait(bar(C::B_DRAIN), 0);
            }
        }
    } else {
        if (!skip) {
            // ------------------------------------------------------------ softmax warpgroups
            const int t = (warp - 4) >> 2;
            const int wq = warp & 3;                 // TMEM lane quarter of this warp
            const int r = wq * 32 + lane;            // row within the tile
            const int row = q0 + kTile * t + r;      // row within the head
            const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
            const uint32_t s_addr = tmem + lane_off + C::s_col(t);
            const uint32_t o_addr = tmem + lane_off + C::o_col(t);
            const float cs = args.scale_log2;
            float m_ref = -INFINITY;  // reference max (log2 domain) shared by O and l
            float l = 0.f;            // sum of p (fp32): the normaliser inside lse
            float lb = 0.f;           // sum of p as rounded for the PV MMA: normalises O
            bool ok = true;
            for (int j = 0; j < nkv[t]; ++j) {
                ok = __all_sync(0xffffffffu, wait_bar(wc, bar(C::B_SFULL + t), j & 1));
                if (!ok) break;
                tc_fence_after();
                if constexpr (SPARSE) {
                    if (((blist[j] >> (14 + t)) & 1) == 0) {
                        // this tile drops the block: P = 0, row state unchanged
                        uint32_t zz[32];
    #pragma unroll
                        for (int e = 0; e < 32; ++e) zz[e] = 0u;
                        tmem_st32(s_addr, zz);
                        tmem_st32(s_addr + 32, zz);
                        tmem_st_wait();
                        tc_fence_before();
                        mbar_arrive(bar(C::B_PFULL + t));
                        continue;
                    }
                }
                float sv[128];
                tmem_ld_sync(s_addr, sv);
                // mask: key tail (keys >= Nk) and, on the diagonal block, keys > row + koff
                const int kb = kblk(j);
                int limit = Nk - kb * kTile;
                if (CAUSAL) limit = min(limit, row + koff - kb * kTile + 1);
                if (limit < kTile) {
    #pragma unroll
                    for (int c = 0; c < kTile; ++c)
                        if (c >= limit) sv[c] = -INFINITY;
                }
                // row max: four independent chains of 3-input max
                float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
    #pragma unroll
                for (int c = 4; c < kTile; c += 8) {
                    mx0 = max3(mx0, sv[c], sv[c + 1]);
                    mx1 = max3(mx1, sv[c + 2], sv[c + 3]);
                    mx2 = max3(mx2, sv[c + 4], sv[c + 5]);
                    mx3 = max3(mx3, sv[c + 6], sv[c + 7]);
                }
                mx0 = max3(mx0, sv[124], sv[125]);
                mx1 = max3(mx1, sv[126], sv[127]);
                const float m_new = fmaxf(m_ref, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * cs);
                const bool move = m_new > m_ref + 8.0f;
                float alpha = 1.0f;
                if (move) {
                    alpha = ex2_approx(m_ref - m_new);  // 0 on the first block
                    l *= alpha;
                    lb *= alpha;
                    m_ref = m_new;
                }
                // p = exp2(s tau log2e - m_ref), two columns per FMA / add instruction
                const uint64_t cs2 = f2_pack(cs, cs);
                // (packed batches: a row that sees no key keeps m_ref = -inf; its p
                // must come out 0, not exp2(-inf + inf))
                const float nm = (VARLEN && m_ref == -INFINITY) ? 0.f : -m_ref;
                const uint64_t nm2 = f2_pack(nm, nm);
                uint64_t sum2 = f2_pack(0.f, 0.f);
                float sumb0 = 0.f, sumb1 = 0.f;
                // TRAIN also sums the rounded p (two widening adds per pair);
                // it stores P in 16-column pieces (32 values) to keep that in registers.
                constexpr int PW = TRAIN ? 32 : 64;  // p values per TMEM store
    #pragma unroll
                for (int h = 0; h < 128 / PW; ++h) {
                    uint32_t pk[PW / 2];
                    // dropout keep bytes of these columns: one generator call per lane
                    // and 16-column group, exchanged so that each lane holds its row's
                    // bytes (patch row = its row % 4); then 0xFF per kept byte
                    uint32_t keep4[PW / 16][4];
                    if constexpr (DROPOUT) {
                        const uint32_t rp = static_cast<uint32_t>((q0 + kTile * t + 32 * wq) >> 2) + (lane >> 2);
                        const uint32_t t4 = args.drop.drop_t * 0x01010101u;
    #pragma unroll
                        for (int g = 0; g < PW / 16; ++g) {
                            const int m = (PW / 16) * h + g;
                            const uint4 w = philox4x32_10(
                                make_uint4(static_cast<uint32_t>(j * 32 + (lane & 3) + 4 * m), rp,
                                           static_cast<uint32_t>(bh), args.drop.offset),
                                args.drop.seed_lo, args.drop.seed_hi);
                            exchange_patch_words(w, lane, keep4[g]);
    #pragma unroll
                            for (int cpp = 0; cpp < 4; ++cpp) keep4[g][cpp] = __vcmpltu4(keep4[g][cpp], t4);
                        }
                    }
    #pragma unroll
                    for (int e = 0; e < PW / 2; ++e) {
                        const uint64_t arg = f2_fma(f2_pack(sv[PW * h + 2 * e], sv[PW * h + 2 * e + 1]), cs2, nm2);
                        float a0, a1;
                        f2_unpack(arg, a0, a1);
                        const float p0 = ex2_approx(a0);
                        const float p1 = ex2_approx(a1);
                        sum2 = f2_add(sum2, f2_pack(p0, p1));
                        pk[e] = pack2<BF16>(p0, p1);
                        if constexpr (TRAIN) add_halves<BF16>(sumb0, sumb1, pk[e]);
                        if constexpr (DROPOUT)   // zero the dropped halves; lb keeps them
                            pk[e] &= __byte_perm(keep4[e / 8][(e % 8) / 2], 0u, (e & 1) ? 0x3322 : 0x1100);
                    }
                    if constexpr (TRAIN)
                        tmem_st16(s_addr + PW / 2 * h, pk);
                    else
                        tmem_st32(s_addr + PW / 2 * h, pk);
                }
                float sum0, sum1;
                f2_unpack(sum2, sum0, sum1);
                l += sum0 + sum1;
                if constexpr (TRAIN) lb += sumb0 + sumb1;
                // Rescale O after the P stores, when the S registers are dead.  O holds
                // P V up to block j-1 (S of block j was committed after that MMA).
                if (j > 0 && __any_sync(0xffffffffu, move)) {
    #pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t orr[32];
                        tmem_ld_sync(o_addr + c, orr);
    #pragma unroll
                        for (int e = 0; e < 32; ++e)
                            orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(o_addr + c, orr);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(C::B_PFULL + t));
            }
            // ------------------------------------------------------------ epilogue
            // The 16-bit O leaves through the tile's Q buffer (free once the tile's
            // last MMA has completed), written out with TMA tensor stores: each
            // thread stages its row in the 128-byte-swizzled box layout and the
            // warpgroup's first thread issues the stores once all rows are in.  The
            // fp32 O (TRAIN) goes straight from TMEM to global memory, read in the
            // 16-lane x 256-bit shape so that every warp-wide store covers whole
            // 32-byte sectors of the rows.
            if (ok && nkv[t] > 0) ok = __all_sync(0xffffffffu, wait_bar(wc, bar(C::B_OFULL + t), 0));
            if (ok && nkv[t] > 0) {
                tc_fence_after();
                // TRAIN normalises O by the sum of the rounded p that actually
                // multiplied V, so each fp32 output row is a convex combination of V
                // rows (weights summing to 1) and rowsum(dO o O) matches the P the
                // backward recomputes; lse keeps the exact sum either way.
                const float den = TRAIN ? lb : l;
                // (block-sparse: a row whose kept tiles were all above the
                // diagonal has an empty softmax, O = 0)
                // (dropout: the kept weights are scaled by 256 / t)
                const float inv_l = ((SPARSE || VARLEN) && !(den > 0.f)) ? 0.f
                                    : (DROPOUT ? args.drop.drop_scale : 1.0f) / den;
                const bool issuer = (warp & 3) == 0 && lane == 0;
                const uint32_t stage = sbase + C::Q_OFF + t * C::TILE_BYTES;
                uint8_t* stage_row = smem + C::Q_OFF + t * C::TILE_BYTES + r * 128;
                const int row0 = q0 + kTile * t;
                if (VARLEN && row0 + kTile > N) {
                    // The last, partial tile of a sequence: a TMA box would also cover
                    // the first rows of the next sequence, so each thread stores its
                    // own row (rows past the sequence are not written).
                    const size_t rbase = (static_cast<size_t>(tok0 + row) * args.H + hq) * D;
    #pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t orr[32];
                        tmem_ld_sync(o_addr + c, orr);
                        if (row < N) {
                            if constexpr (TRAIN) {
    #pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    *reinterpret_cast<float4*>(args.o32 + rbase + c + 4 * e) =
                                        make_float4(__uint_as_float(orr[4 * e]) * inv_l,
                                                    __uint_as_float(orr[4 * e + 1]) * inv_l,
                                                    __uint_as_float(orr[4 * e + 2]) * inv_l,
                                                    __uint_as_float(orr[4 * e + 3]) * inv_l);
                            }
                            uint32_t pk[16];
    #pragma unroll
                            for (int e = 0; e < 16; ++e)
                                pk[e] = pack2<BF16>(__uint_as_float(orr[2 * e]) * inv_l,
                                                    __uint_as_float(orr[2 * e + 1]) * inv_l);
    #pragma unroll
                            for (int e = 0; e < 4; ++e)
                                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + rbase + c + 8 * e) =
                                    make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                        }
                    }
                }
                if (ok && !(VARLEN && row0 + kTile > N)) {
                    // all D columns of the 16-bit O: boxes of 64 columns
    #pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t orr[32];
                        tmem_ld_sync(o_addr + c, orr);
                        uint32_t pk[16];
    #pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack2<BF16>(__uint_as_float(orr[2 * e]) * inv_l,
                                                __uint_as_float(orr[2 * e + 1]) * inv_l);
                        uint8_t* box_row = stage_row + (c / 64) * kBoxBytes;
                        const int ch0 = (c % 64) / 8;   // 16-byte chunks of this 32-column piece
    #pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            *reinterpret_cast<uint4*>(box_row + (((ch0 + v4) ^ (r & 7)) * 16)) =
                                make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(bar(C::B_EPI_STAGED + t));
                    if (issuer && wait_bar(wc, bar(C::B_EPI_STAGED + t), 0)) {
                        for (int b = 0; b < D / 64; ++b)
                            tma_store_3d(&tm_o, stage + b * kBoxBytes, 64 * b, tok0 + row0, hq);
                        bulk_commit_group();
                        bulk_wait_group_read<0>();
                    }
                }
                if (TRAIN && ok && !(VARLEN && row0 + kTile > N)) {
                    // fp32 O: thread t of the warp holds, per 16-lane half hh and
                    // 64-column piece, rows 16 hh + t / 4 and 16 hh + t / 4 + 8 of the
                    // warp's 32 at columns 2 (t % 4) + {0, 1} of each 8-column group;
                    // the normaliser of a row comes from the thread that owns it
    #pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
    #pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int src = 16 * hh + (lane >> 2) + 8 * rr;       // row within the warp
                            const float inv = __shfl_sync(0xffffffffu, inv_l, src);
                            const int grow = row0 + 32 * wq + src;
                            float* dst = args.o32 +
                                         (VARLEN ? (static_cast<size_t>(tok0 + grow) * args.H + hq) * D
                                                 : (static_cast<size_t>(bh) * N + grow) * D) +
                                         2 * (lane & 3);
    #pragma unroll
                            for (int cc = 0; cc < D; cc += 64) {
                                uint32_t v[32];
                                tmem_ld_16x256b_x8(tmem + (static_cast<uint32_t>(32 * wq + 16 * hh) << 16) +
                                                       C::o_col(t) + cc, v);
                                if (grow < N) {
    #pragma unroll
                                    for (int g = 0; g < 8; ++g)
                                        *reinterpret_cast<float2*>(dst + cc + 8 * g) =
                                            make_float2(__uint_as_float(v[4 * g + 2 * rr]) * inv,
                                                        __uint_as_float(v[4 * g + 2 * rr + 1]) * inv);
                                }
                            }
                        }
                    }
                }
                // The stores only have to finish reading shared memory before the
                // CTA exits (done above); their global writes complete with the
                // kernel, and waiting for them here kept the next CTA off the SM.
                if (row < N)
                    args.lse[static_cast<size_t>(bh) * (VARLEN ? args.max_seqlen : N) + row] =
                        (((SPARSE || VARLEN) && !(l > 0.f)) ? -INFINITY : (m_ref + __log2f(l)) * kLn2);
            }
            if (VARLEN && ok && nkv[t] == 0 && row < N) {
                // packed batch, keys shorter than the queries: every row of this tile
                // precedes the first visible key (the other tile has work), O = 0,
                // lse = -inf, each thread its own row
                const size_t rbase = (static_cast<size_t>(tok0 + row) * args.H + hq) * D;
                for (int c = 0; c < D; c += 8)
                    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + rbase + c) = make_uint4(0u, 0u, 0u, 0u);
                if (TRAIN)
                    for (int c = 0; c < D; c += 4)
                        *reinterpret_cast<float4*>(args.o32 + rbase + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                args.lse[static_cast<size_t>(bh) * args.max_seqlen + row] = -INFINITY;
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

template <int D, bool CAUSAL, bool BF16, bool TRAIN, bool VARLEN, bool SPARSE = false,
          bool DROPOUT = false>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& to,
                                const CUtensorMap& to32, const FwdArgs& a, int BH,
                                cudaStream_t stream) {
    using C = FwdCfg<D>;
    auto kern = attn_fwd_kernel<D, CAUSAL, BF16, TRAIN, VARLEN, SPARSE, DROPOUT>;
    constexpr int smem = SPARSE ? C::SMEM_SPARSE : C::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid = VARLEN ? head_major_grid(a.num_qblocks, BH)
                             : group_grid(a.num_qblocks, BH, a.head_group > 0 ? a.head_group : BH);
    kern<<<grid, C::THREADS, smem, stream>>>(tq, tk, tv, to, to32, a);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& to32, const FwdArgs& a, int BH,
                       int d, bool causal, bool bf16, cudaStream_t stream) {
    const bool varlen = a.cu_seqlens != nullptr;
    const bool sparse = a.block_mask != nullptr;
    const bool dropout = a.drop.drop_t > 0 && a.drop.drop_t < 256;   // training path, dense only
    if (dropout && (varlen || sparse || a.o32 == nullptr)) return cudaErrorInvalidValue;
#define ATTN_FWD_CASE(D_, C_, B_)                                                                   \
    if (d == D_ && causal == C_ && bf16 == B_) {                                                    \
        if (dropout)                                                                                \
            return launch_fwd_t<D_, C_, B_, true, false, false, true>(tq, tk, tv, to, to32, a, BH, stream); \
        if (sparse)                                                                                 \
            return a.o32 != nullptr ? launch_fwd_t<D_, C_, B_, true, false, true>(tq, tk, tv, to, to32, a, BH, stream) \
                                    : launch_fwd_t<D_, C_, B_, false, false, true>(tq, tk, tv, to, to32, a, BH, stream); \
        if (varlen)                                                                                 \
            return a.o32 != nullptr ? launch_fwd_t<D_, C_, B_, true, true>(tq, tk, tv, to, to32, a, BH, stream) \
                                    : launch_fwd_t<D_, C_, B_, false, true>(tq, tk, tv, to, to32, a, BH, stream); \
        return a.o32 != nullptr ? launch_fwd_t<D_, C_, B_, true, false>(tq, tk, tv, to, to32, a, BH, stream) \
                                : launch_fwd_t<D_, C_, B_, false, false>(tq, tk, tv, to, to32, a, BH, stream); \
    }
    ATTN_FWD_CASE(64, false, true)
    ATTN_FWD_CASE(64, true, true)
    ATTN_FWD_CASE(128, false, true)
    ATTN_FWD_CASE(128, true, true)
    ATTN_FWD_CASE(64, false, false)
    ATTN_FWD_CASE(64, true, false)
    ATTN_FWD_CASE(128, false, false)
    ATTN_FWD_CASE(128, true, false)
#undef ATTN_FWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace attn
