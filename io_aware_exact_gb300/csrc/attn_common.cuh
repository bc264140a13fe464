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
    // Block-sparse layout (nullptr: none): one byte per 128 x 128 tile
    // (query block, key block) at block_mask + bh * mask_head_stride, row-major
    // with mask_cols = ceil(N / 128) columns; zero drops the tile.
    const uint8_t* block_mask;
    long long mask_head_stride;
    int mask_cols;
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
    // block-sparse layout as in FwdArgs (nullptr: none)
    const uint8_t* block_mask;
    long long mask_head_stride;
    int mask_cols;
    // fp32 gradient outputs (dense layout, general kernel), nullptr: 16-bit dk, dv.
    // dk32 / dv32 [B*Hkv, N, d] are overwritten, or added to when acc32 != 0.
    float* dk32;
    float* dv32;
    int acc32;
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

inline int device_sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 152;
    }
    return n;
}

// K / V head of (batch, query head) bh when groups of H / Hkv query heads share one
__device__ __forceinline__ int kv_head(int bh, int H, int Hkv) {
    return (bh / H) * Hkv + (bh % H) / (H / Hkv);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
}

}  // namespace attn
