// attn_common.cuh - shared declarations of the CUDA attention library.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Tile geometry shared by forward and backward: 128 query rows x 128 keys per
// MMA tile; tiles are stored in shared memory as 64-column (128-byte) boxes
// with the 128-byte swizzle, which is the layout the TMA box writes and the
// tensor-core descriptors read.
constexpr int kTile = 128;
constexpr int kBoxCols = 64;
constexpr int kBoxBytes = kTile * kBoxCols * 2;  // 16 KB

// Block-sparse layouts: a CTA lists the tiles it keeps in shared memory, at
// most this many (N <= 384 * 128 = 49,152); list entries are 16-bit.
constexpr int kMaxSparseBlocks = 384;

// Dropout (training forward and backward): the keep mask is regenerated
// from (seed, offset) in both passes, never stored.  Element (i, j) of head
// bh keeps iff byte j % 4 of word i % 4 of Philox4x32-10 with counter
// (j / 4, i / 4, bh, offset) and key (seed_lo, seed_hi) is below drop_t; kept
// weights are scaled by drop_scale = 256 / drop_t.
struct DropoutArgs {
    uint32_t seed_lo, seed_hi, offset;
    uint32_t drop_t;       // 1..255 (256, no dropout, uses the kernels without it)
    float drop_scale;      // 256 / drop_t
};

struct FwdArgs {
    void* o;               // [B*H, N, d] 16-bit, written
    float* o32;            // [B*H, N, d] fp32 copy of O for the backward, or nullptr
    float* lse;            // [B*H, N] fp32, written (natural log, scale inside)
    int* status;           // device status word
    int N;                 // sequence length
    int BH;                // batch * query heads
    int H;                 // query heads
    int Hkv;               // key / value heads (H is a multiple; query head h reads K/V head h / (H / Hkv))
    int num_qblocks;       // ceil(N / 256): CTAs per head
    int head_group;        // dense grid in head groups (x = head in group, y = block, z = group); 0: plain
    // Packed variable-length batch (nullptr: dense [B,H,N,d]): sequence b is
    // tokens [cu_seqlens[b], cu_seqlens[b+1]) of [total, H, d]; N = max_seqlen
    // then, and lse is [B, H, max_seqlen].
    const int* cu_seqlens;
    int total;
    int max_seqlen;
    // Keys of a different length (nullptr: the key rows of sequence b are its
    // query rows): sequence b's keys / values are rows [cu_seqlens_k[b],
    // cu_seqlens_k[b+1]) of the [total_k, Hkv, d] K and V, and with a causal
    // mask key j is visible to query i iff j <= i + Lk - Lq (bottom-right).
    const int* cu_seqlens_k;
    int total_k;
    int max_seqlen_k;
    // Block-sparse layout (nullptr: none): one byte per 128 x 128 tile
    // (query block, key block) at block_mask + bh * mask_head_stride, row-major
    // with mask_cols = ceil(N / 128) columns; zero drops the tile.
    const uint8_t* block_mask;
    long long mask_head_stride;
    int mask_cols;
    DropoutArgs drop;      // used by the dropout instantiations only
    float scale_log2;      // softmax scale * log2(e)
    unsigned int wait_polls;   // try_wait polls before a wait gives up (about 2 us each)
};

struct BwdArgs {
    const float* lse;      // [B*H, N]
    const float* D;        // [B*H, N]
    float* dq_accum;       // [B*H, N, d] fp32 (reduced into through a tensor map)
    void* dk;              // [B*H, N, d] 16-bit
    void* dv;              // [B*H, N, d] 16-bit
    int* status;
    int N;
    int BH;                // batch * query heads
    int H;                 // query heads
    int Hkv;               // key / value heads (grid: batch * Hkv); query heads per group H / Hkv
    int BHkv;              // batch * key / value heads
    int head_group;        // dense grid in head groups (x = head in group, y = block, z = group); 0: plain
    int num_kvblocks;      // ceil(N / 128)
    // packed variable-length batch as in FwdArgs (nullptr: dense); D is then
    // [total, H] (the row order of the packed tensors), lse [B, H, max_seqlen]
    const int* cu_seqlens;
    int total;
    int max_seqlen;
    // keys of a different length as in FwdArgs (nullptr: same as the queries);
    // K, V, dK, dV are then [total_k, Hkv, d]
    const int* cu_seqlens_k;
    int total_k;
    int max_seqlen_k;
    // block-sparse layout as in FwdArgs (nullptr: none)
    const uint8_t* block_mask;
    long long mask_head_stride;
    int mask_cols;
    // fp32 gradient outputs (dense layout, general kernel), nullptr: 16-bit dk, dv.
    // dk32 / dv32 [B*Hkv, N, d] are overwritten, or added to when acc32 != 0.
    float* dk32;
    float* dv32;
    int acc32;
    // grouped heads, dense layout: the group's query heads are split over
    // `splits` CTAs per (K / V head, key block); split s writes its share of
    // dK, dV (fp32) at dk32 / dv32 + s * split_stride, summed afterwards
    int splits;
    long long split_stride;
    DropoutArgs drop;      // used by the dropout instantiations only
    float scale;           // softmax scale (tau)
    float scale_log2;      // tau * log2(e)
    unsigned int wait_polls;   // try_wait polls before a wait gives up (about 2 us each)
};

struct DsumArgs {
    const float* lse;      // [B*H, N]
    float* D;              // [B*H, N], written: sum_j P_ij dP_ij
    float* dq_accum;       // [B*H, N, d] fp32, zeroed
    int* status;
    int N;
    int BH;                // batch * query heads
    int H;                 // query heads
    int Hkv;               // key / value heads
    float scale_log2;      // tau * log2(e)
    unsigned int wait_polls;   // try_wait polls before a wait gives up (about 2 us each)
};

struct PreO32Args {
    const float* o32;      // [B*H, N, d] fp32 O from attn_fwd_train
    const void* dO;        // [B*H, N, d] 16-bit
    float* D;              // [B*H, N]
    float* dq_accum;       // [B*H, N, d] fp32, zeroed
    long long rows;        // B*H*N
    int d;
};

struct DqConvertArgs {
    const float* dq_accum;  // [B*H, N, d]
    void* dq;               // [B*H, N, d] 16-bit
    long long elems;        // B*H*N*d
    float scale;            // tau
};

struct SplitSumArgs {
    const float* part;      // [splits][elems] fp32 shares
    void* out;              // [elems] 16-bit sum
    long long elems;        // multiple of 8
    int splits;
};

struct MergeArgs {
    float* o_acc;           // [rows, d] fp32 running output, merged in place
    float* lse_acc;         // [rows] running logsumexp, merged in place
    const float* o_part;    // [rows, d] fp32 partial output
    const float* lse_part;  // [rows] partial logsumexp
    void* o_out;            // [rows, d] 16-bit copy of the merged output, or nullptr
    long long rows;
    int d;
};

// Launchers (defined in the kernel translation units).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const CUtensorMap& to32, const FwdArgs& a, int BH,
                       int d, bool causal, bool bf16, cudaStream_t stream);
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                       const CUtensorMap& tdv, const BwdArgs& a, int BH, int d, bool causal,
                       bool bf16, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const DsumArgs& a, int BH, int d, bool causal,
                            bool bf16, cudaStream_t stream);
cudaError_t launch_bwd_preprocess_o32(const PreO32Args& a, bool bf16, cudaStream_t stream);
cudaError_t launch_dq_convert(const DqConvertArgs& a, bool bf16, cudaStream_t stream);
cudaError_t launch_merge(const MergeArgs& a, bool bf16, cudaStream_t stream);
cudaError_t launch_split_sum(const SplitSumArgs& a, bool bf16, cudaStream_t stream);


// Grid layouts of the attention kernels.  Plain: x = (batch, head), y/z =
// block index within a head.  Launch order is x fastest, so every head's
// heaviest causal block is scheduled before any lighter one (longest work
// first); y is capped at the hardware limit and z extends it.  The index math
// is a few reads of blockIdx and no division: the backward runs at its
// register limit, and a division-based mapping cost it about 4%.
constexpr int kMaxGridY = 65535;

inline dim3 lpt_grid(int blocks_per_head, int BH) {
    const int gy = blocks_per_head < kMaxGridY ? blocks_per_head : kMaxGridY;
    return dim3(BH, gy, (blocks_per_head + gy - 1) / gy);
}

// Head-major variant: x = block index within the head (0 launched first), y
// (and z beyond 65,535) = head, so all blocks of one head run close together.
inline dim3 head_major_grid(int blocks_per_head, int heads) {
    const int gy = heads < kMaxGridY ? heads : kMaxGridY;
    return dim3(blocks_per_head, gy, (heads + gy - 1) / gy);
}

// Head groups: x = head within a group of G heads, y = block rank, z = group,
// so the blocks of G heads run together, longest work first within the group.
// Needs G to divide the head count and blocks_per_head <= 65,535.
inline dim3 group_grid(int blocks_per_head, int heads, int G) {
    return dim3(G, blocks_per_head, heads / G);
}

// Re-read bytes a head group may hold (L2 is 126 MB): measured on the causal
// B=2 H=16 N=8192 d=128 workload, groups of 8 heads beat 2, 4, 16 and all 32.
constexpr long long kFwdGroupBytes = 32ll << 20;
constexpr long long kBwdGroupBytes = 64ll << 20;
int head_group_for(int heads, int blocks_per_head, long long bytes_per_head, long long budget);

// Block index within the head (0 = first launched); >= blocks_per_head only
// for padding CTAs of the last z-slice.
__device__ __forceinline__ int grid_block() {
    return static_cast<int>(blockIdx.z) * static_cast<int>(gridDim.y) + static_cast<int>(blockIdx.y);
}

// SM count of the current device (cached per device index; thread-safe).
int device_sm_count();

// K / V head of (batch, query head) bh when groups of H / Hkv query heads share one
__device__ __forceinline__ int kv_head(int bh, int H, int Hkv) {
    return (bh / H) * Hkv + (bh % H) / (H / Hkv);
}

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11): each round maps (c0, c1, c2, c3) with
// key (k0, k1) to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
// lo(M0 c0)), and the key is bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

__device__ __forceinline__ uint32_t sel4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, int i) {
    return i == 0 ? a : i == 1 ? b : i == 2 ? c : d;
}

// Keep masks of one 4 x 4 patch exchanged inside a group of four lanes.
// Lane L of the group computes the patch at position (L & 3) + 4m of a row of
// patches (four words w, word a = patch row a, byte b = patch column b), and
// needs word `want` of every patch of that row: in round rr it receives, from
// lane (L & 3) + rr of its group, the word of patch ((L & 3) + rr) & 3 + 4m
// (the source sends its word (its lane - rr) & 3).  Returned in rv[cpp] for
// patch cpp + 4m, cpp = 0..3.
__device__ __forceinline__ void exchange_patch_words(uint4 w, int lane, uint32_t (&rv)[4]) {
    const int l = lane & 3;
    uint32_t got[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const uint32_t send = sel4(w.x, w.y, w.z, w.w, (l - rr) & 3);
        got[rr] = __shfl_sync(0xffffffffu, send, (lane & ~3) | ((l + rr) & 3));
    }
#pragma unroll
    for (int cpp = 0; cpp < 4; ++cpp) rv[cpp] = sel4(got[0], got[1], got[2], got[3], (cpp - l) & 3);
}

// 4 x 4 byte transpose: result word b holds byte b of w.x, w.y, w.z, w.w.
__device__ __forceinline__ uint4 transpose_bytes(uint4 w) {
    const uint32_t t0 = __byte_perm(w.x, w.y, 0x5140), t1 = __byte_perm(w.x, w.y, 0x7362);
    const uint32_t t2 = __byte_perm(w.z, w.w, 0x5140), t3 = __byte_perm(w.z, w.w, 0x7362);
    return make_uint4(__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                      __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632));
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
}

}  // namespace attn
