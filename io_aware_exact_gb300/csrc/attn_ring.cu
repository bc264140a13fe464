// attn_ring.cu - element-wise kernels that combine partial attention results.
//
// Attention over a sequence split into key / value chunks (ring or
// context-parallel attention) computes, for each chunk, a partial output
// normalised over that chunk's keys and the chunk's logsumexp.  Two partial
// states of one query row combine exactly (sj-techlog "FlashAttention 원 논문
// 해부", section "두 tile을 한 row로 합치는 식": rescale both by exp of their
// statistic minus the new maximum and renormalise).  With normalised outputs
// and logsumexps L1, L2 that is
//
//   L = log(exp(L1) + exp(L2)),   O = exp(L1 - L) O1 + exp(L2 - L) O2,
//
// evaluated here with the larger statistic subtracted first.  A partial with
// L = -inf (no visible key) carries weight 0; two of them give O = 0, L = -inf.
//
// The kernels are memory-bound: one pass over the rows, 16-byte accesses.
#include "attn_common.cuh"

namespace attn {

// One warp covers 32 / TPR rows per step (TPR = d / 4 lanes per row, one
// float4 each); the loop bound is warp-uniform so that the lanes of a row can
// synchronise between reading the two statistics and writing the merged one.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const MergeArgs a) {
    constexpr int TPR = D / 4;
    constexpr int ROWS_PER_WARP = 32 / TPR;
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int c = (lane % TPR) * 4;
    for (long long r0 = warp * ROWS_PER_WARP; r0 < a.rows; r0 += nwarps * ROWS_PER_WARP) {
        const long long row = r0 + lane / TPR;
        const bool valid = row < a.rows;
        float l1 = -INFINITY, l2 = -INFINITY;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
        if (valid) {
            l1 = a.lse_acc[row];
            l2 = a.lse_part[row];
            x = *reinterpret_cast<const float4*>(a.o_acc + row * D + c);
            y = *reinterpret_cast<const float4*>(a.o_part + row * D + c);
        }
        __syncwarp();
        const float mx = fmaxf(l1, l2);
        float w1 = 0.f, w2 = 0.f, l = -INFINITY;
        if (mx != -INFINITY) {
            const float e1 = expf(l1 - mx), e2 = expf(l2 - mx);
            const float s = e1 + e2;
            l = mx + logf(s);
            w1 = e1 / s;
            w2 = e2 / s;
        }
        if (valid) {
            const float4 o = make_float4(w1 * x.x + w2 * y.x, w1 * x.y + w2 * y.y,
                                         w1 * x.z + w2 * y.z, w1 * x.w + w2 * y.w);
            *reinterpret_cast<float4*>(a.o_acc + row * D + c) = o;
            if (a.o_out != nullptr)
                *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.o_out) + row * D + c) =
                    make_uint2(pack2<BF16>(o.x, o.y), pack2<BF16>(o.z, o.w));
            if (c == 0) a.lse_acc[row] = l;
        }
    }
}

// out = sum over s of part[s], rounded to 16 bits; eight elements per step.
template <bool BF16>
__global__ void __launch_bounds__(256) attn_split_sum_kernel(const SplitSumArgs a) {
    const long long n8 = a.elems / 8;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += stride) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
        for (int s = 0; s < a.splits; ++s) {
            const float4* p = reinterpret_cast<const float4*>(a.part + s * a.elems) + 2 * i;
            const float4 u = p[0], w = p[1];
            x.x += u.x; x.y += u.y; x.z += u.z; x.w += u.w;
            y.x += w.x; y.y += w.y; y.z += w.z; y.w += w.w;
        }
        reinterpret_cast<uint4*>(a.out)[i] = make_uint4(pack2<BF16>(x.x, x.y), pack2<BF16>(x.z, x.w),
                                                        pack2<BF16>(y.x, y.y), pack2<BF16>(y.z, y.w));
    }
}

static long long elementwise_blocks(long long work_items) {
    long long blocks = (work_items + 255) / 256;
    const long long cap = static_cast<long long>(device_sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : blocks;
}

cudaError_t launch_merge(const MergeArgs& a, bool bf16, cudaStream_t stream) {
    const long long blocks = elementwise_blocks(a.rows * (a.d / 4));
#define ATTN_MERGE_CASE(D_, B_) \
    if (a.d == D_ && bf16 == B_) attn_merge_kernel<B_, D_><<<blocks, 256, 0, stream>>>(a); else
    ATTN_MERGE_CASE(64, true)
    ATTN_MERGE_CASE(128, true)
    ATTN_MERGE_CASE(64, false)
    ATTN_MERGE_CASE(128, false)
    return cudaErrorInvalidValue;
#undef ATTN_MERGE_CASE
    return cudaGetLastError();
}

cudaError_t launch_split_sum(const SplitSumArgs& a, bool bf16, cudaStream_t stream) {
    const long long blocks = elementwise_blocks(a.elems / 8);
    if (bf16) attn_split_sum_kernel<true><<<blocks, 256, 0, stream>>>(a);
    else attn_split_sum_kernel<false><<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace attn
