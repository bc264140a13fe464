// attn_api.cu - C ABI entry points: argument checks, TMA tensor maps, launches.
//
// The host layer plays the part of the reference's C++ dispatcher (sj-techlog
// "FlashAttention 원 논문 해부", section "3. C++ dispatcher는 N² buffer를 언제
// 만들지 명시적으로 고른다": device/shape/head-size checks, then a launch on
// the caller's stream) but allocates nothing: every buffer is the caller's.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/attn.h"
#include "attn_common.cuh"

namespace attn {

// Head group size for a dense grid: the largest divisor G of `heads` whose G
// heads' re-read bytes (bytes_per_head) fit in `budget`, raised if needed so
// that a group still holds two waves of CTAs; 0 (plain order) when that is all
// heads or the grid would not fit.
int head_group_for(int heads, int blocks_per_head, long long bytes_per_head, long long budget) {
    if (blocks_per_head > kMaxGridY || heads <= 1) return 0;
    int g = 1;
    for (int c = heads; c >= 1; --c)
        if (heads % c == 0 && static_cast<long long>(c) * bytes_per_head <= budget) { g = c; break; }
    const long long min_ctas = 2ll * device_sm_count();
    while (g < heads && static_cast<long long>(g) * blocks_per_head < min_ctas) {
        int c = g + 1;
        while (heads % c != 0) ++c;
        g = c;
    }
    return g >= heads ? 0 : g;
}

// Device status word written by kernels whose bounded waits run out.
__device__ int g_status;

namespace {

// try_wait polls before a bounded wait gives up: an unsuccessful poll suspends
// the thread for about 2 us, so this is about 2 s.
constexpr unsigned int kDefaultWaitPolls = 1000000u;
// Longest dense sequence: the forward's grid holds at most 65,535 blocks of
// 256 query rows in one dimension.
constexpr int kMaxN = (1 << 24) - 256;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct DevInfo {
    bool checked = false;
    bool ok = false;
    int* status = nullptr;
};

constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Validates the current device (sm_103) and returns its status-word address.
int current_device(int** status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return ATTN_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo& di = g_dev[dev];
    if (!di.checked) {
        di.checked = true;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        void* p = nullptr;
        di.ok = (major == 10 && minor == 3) &&
                cudaGetSymbolAddress(&p, g_status) == cudaSuccess && p != nullptr;
        di.status = static_cast<int*>(p);
        if (!di.ok) cudaGetLastError();
    }
    if (!di.ok) return ATTN_ERR_UNSUPPORTED_DEVICE;
    *status = di.status;
    return ATTN_OK;
}

int g_sm_count[kMaxDevices];
std::mutex g_sm_mu;

}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 152;
    }
    std::lock_guard<std::mutex> lk(g_sm_mu);
    if (g_sm_count[dev] <= 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEAD_DIM;
    if (static_cast<long long>(B) * H > 2147483647LL) return ATTN_ERR_INVALID_ARG;
    if (N > kMaxN) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

int check_scale(float s) { return (std::isfinite(s) && s > 0.f) ? ATTN_OK : ATTN_ERR_INVALID_ARG; }

// Grouped K / V heads: Hkv >= 1 and a divisor of H.
int check_kv_heads(int H, int Hkv) { return (Hkv >= 1 && H % Hkv == 0) ? ATTN_OK : ATTN_ERR_INVALID_ARG; }

// 3-D tensor map over a contiguous [BH, N, d] 16-bit array: box = 64 columns x
// 128 rows x 1 head, 128-byte swizzle, zero fill beyond row N of each head.
int make_map(CUtensorMap* m, const void* base, int BH, int N, int d, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return ATTN_ERR_LAUNCH;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                   static_cast<cuuint64_t>(N) * d * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBoxCols), static_cast<cuuint32_t>(kTile), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

// Tile maps, the ones the forward loads Q, K and V through: a 4-D view
// (column within a 64-column half, row, half, head) of the same array, box =
// 64 columns x 128 rows x all d / 64 halves x 1 head, 128-byte swizzle, zero
// fill beyond the last row.  One copy then brings a whole 128 x d tile in the
// layout two 64-column boxes give (each half its own 16 KB swizzled box, the
// halves one after the other).  Copies issued by one thread complete about
// one per 550 cycles whether they carry 16 or 32 KB (measured on GB300), so
// the forward's producer moves K_j and V_j in two copies instead of four.
// The backward keeps the 64-column maps: its reducer thread issues each Q / dO
// reload between the two halves of its dQ reduce-adds, and that kernel
// measured 2.7% faster than a version that reloaded each tile in one copy
// from the producer warp (paired runs on one GB300).
static int encode_tile_map(CUtensorMap* m, const void* base, cuuint64_t rows, cuuint64_t heads, int d,
                           cuuint64_t row_stride, cuuint64_t head_stride, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return ATTN_ERR_LAUNCH;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kBoxCols), rows,
                                static_cast<cuuint64_t>(d / kBoxCols), heads};
    const cuuint64_t strides[3] = {row_stride, static_cast<cuuint64_t>(kBoxCols) * 2, head_stride};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(kBoxCols), static_cast<cuuint32_t>(kTile),
                               static_cast<cuuint32_t>(d / kBoxCols), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

// Tile map over a contiguous [BH, N, d] 16-bit array.
int make_tile_map(CUtensorMap* m, const void* base, int BH, int N, int d, bool bf16) {
    return encode_tile_map(m, base, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH), d,
                           static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2, bf16);
}

// 3-D tensor map over a contiguous [BH, N, d] fp32 array (the dQ accumulator,
// the training forward's fp32 O): box = 32 columns (128 bytes) x 128 rows x
// 1 head, 128-byte swizzle; rows beyond N of a head are never written through it.
int make_map_f32(CUtensorMap* m, const void* base, int BH, int N, int d) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return ATTN_ERR_LAUNCH;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                   static_cast<cuuint64_t>(N) * d * 4};
    const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(kTile), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

int map_launch(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH; }

// Block-sparse layout checks: a mask is given, one query head per K / V
// head, N within the shared-memory list, and per-head masks (stride > 0) do
// not overlap.
int check_sparse(const void* block_mask, long long mask_stride, int H, int Hkv, int N) {
    if (!block_mask || H != Hkv || N > kMaxSparseBlocks * kTile || mask_stride < 0)
        return ATTN_ERR_INVALID_ARG;
    const long long nb = (N + kTile - 1) / kTile;
    if (mask_stride != 0 && mask_stride < nb * nb) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

// Dropout settings from the drop probability: keep iff a random byte is below
// t = 256 (1 - p) rounded half to even, clamped to [1, 256]; t = 256 keeps all.
int make_dropout(float p_drop, unsigned long long seed, unsigned int offset, DropoutArgs* out) {
    if (!std::isfinite(p_drop) || p_drop < 0.f || p_drop >= 1.f) return ATTN_ERR_INVALID_ARG;
    double t = std::nearbyint(256.0 * (1.0 - static_cast<double>(p_drop)));
    t = t < 1.0 ? 1.0 : (t > 256.0 ? 256.0 : t);
    out->seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFull);
    out->seed_hi = static_cast<uint32_t>(seed >> 32);
    out->offset = offset;
    out->drop_t = static_cast<uint32_t>(t);
    out->drop_scale = static_cast<float>(256.0 / t);
    return ATTN_OK;
}

// Variants of the forward beyond the dense path (defaults: none).
struct FwdOptions {
    const void* block_mask = nullptr;   // block-sparse layout
    long long mask_stride = 0;
    const DropoutArgs* drop = nullptr;  // dropout on P
};

// Variants of the backward beyond the dense path (defaults: none).
struct BwdOptions {
    const void* block_mask = nullptr;   // block-sparse layout
    long long mask_stride = 0;
    float* dk32 = nullptr;              // fp32 dK, dV written (or added, acc32) instead of dk, dv
    float* dv32 = nullptr;
    int acc32 = 0;
    const DropoutArgs* drop = nullptr;  // dropout on P
    int splits = 1;                     // grouped heads: query-head shares per group
    float* split_part = nullptr;        // their fp32 dK, dV shares
};

FwdOptions sparse_fwd(const void* mask, long long stride) {
    FwdOptions o;
    o.block_mask = mask;
    o.mask_stride = stride;
    return o;
}

BwdOptions sparse_bwd(const void* mask, long long stride) {
    BwdOptions o;
    o.block_mask = mask;
    o.mask_stride = stride;
    return o;
}

BwdOptions f32_bwd(float* dk32, float* dv32, int accumulate) {
    BwdOptions o;
    o.dk32 = dk32;
    o.dv32 = dv32;
    o.acc32 = accumulate;
    return o;
}

BwdOptions drop_bwd(const DropoutArgs* drop) {
    BwdOptions o;
    o.drop = drop;
    return o;
}

BwdOptions split_bwd(int splits, float* part) {
    BwdOptions o;
    o.splits = splits;
    o.split_part = part;
    return o;
}

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* o32, float* lse, int B,
             int H, int Hkv, int N, int d, int causal, float scale, void* stream, bool bf16,
             const FwdOptions& opt = FwdOptions()) {
    const void* block_mask = opt.block_mask;
    const long long mask_stride = opt.mask_stride;
    const DropoutArgs* drop = opt.drop;
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (o32 != nullptr && !aligned16(o32)) return ATTN_ERR_MISALIGNED;
    int rc = check_shape(B, H, N, d);
    if (rc) return rc;
    if ((rc = check_kv_heads(H, Hkv))) return rc;
    if ((rc = check_scale(scale))) return rc;
    if (block_mask != nullptr && (rc = check_sparse(block_mask, mask_stride, H, Hkv, N))) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    if ((rc = current_device(&status))) return rc;
    const int BH = B * H, BHkv = B * Hkv;
    CUtensorMap tq, tk, tv, to, to32;
    if ((rc = make_tile_map(&tq, q, BH, N, d, bf16)) || (rc = make_tile_map(&tk, k, BHkv, N, d, bf16)) ||
        (rc = make_tile_map(&tv, v, BHkv, N, d, bf16)) || (rc = make_map(&to, o, BH, N, d, bf16)))
        return rc;
    // the plain forward never touches the fp32 map; it gets a copy of the O map
    if (o32 != nullptr) {
        if ((rc = make_map_f32(&to32, o32, BH, N, d))) return rc;
    } else {
        to32 = to;
    }
    FwdArgs a{};
    a.o = o;
    a.o32 = o32;
    a.lse = lse;
    a.status = status;
    a.N = N;
    a.BH = BH;
    a.H = H;
    a.Hkv = Hkv;
    a.num_qblocks = (N + 2 * kTile - 1) / (2 * kTile);
    // K and V of a head are re-read by each of its query-block CTAs
    a.head_group = head_group_for(BH, a.num_qblocks, 4ll * N * d, kFwdGroupBytes);
    a.block_mask = static_cast<const uint8_t*>(block_mask);
    a.mask_head_stride = mask_stride;
    a.mask_cols = (N + kTile - 1) / kTile;
    if (drop != nullptr) a.drop = *drop;
    a.scale_log2 = scale * kLog2e;
    a.wait_polls = kDefaultWaitPolls;
    return map_launch(launch_fwd(tq, tk, tv, to, to32, a, BH, d, causal != 0, bf16,
                                 static_cast<cudaStream_t>(stream)));
}

int pre_impl(const void* q, const void* k, const void* v, const void* dO, const float* lse,
             float* D, float* dq_accum, int B, int H, int Hkv, int N, int d, int causal,
             float scale, void* stream, bool bf16) {
    if (!q || !k || !v || !dO || !lse || !D || !dq_accum) return ATTN_ERR_INVALID_ARG;
    int rc = check_shape(B, H, N, d);
    if (rc) return rc;
    if ((rc = check_kv_heads(H, Hkv))) return rc;
    if ((rc = check_scale(scale))) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
        !aligned16(D) || !aligned16(dq_accum))
        return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    if ((rc = current_device(&status))) return rc;
    const int BH = B * H, BHkv = B * Hkv;
    CUtensorMap tq, tk, tv, tdo;
    if ((rc = make_map(&tq, q, BH, N, d, bf16)) || (rc = make_map(&tk, k, BHkv, N, d, bf16)) ||
        (rc = make_map(&tv, v, BHkv, N, d, bf16)) || (rc = make_map(&tdo, dO, BH, N, d, bf16)))
        return rc;
    DsumArgs a{};
    a.lse = lse;
    a.D = D;
    a.dq_accum = dq_accum;
    a.status = status;
    a.N = N;
    a.BH = BH;
    a.H = H;
    a.Hkv = Hkv;
    a.scale_log2 = scale * kLog2e;
    a.wait_polls = kDefaultWaitPolls;
    return map_launch(launch_bwd_preprocess(tq, tk, tv, tdo, a, BH, d, causal != 0, bf16,
                                            static_cast<cudaStream_t>(stream)));
}

int pre_o32_impl(const float* o32, const void* dO, float* D, float* dq_accum, int B, int H, int N,
                 int d, void* stream, bool bf16) {
    if (!o32 || !dO || !D || !dq_accum) return ATTN_ERR_INVALID_ARG;
    int rc = check_shape(B, H, N, d);
    if (rc) return rc;
    if (!aligned16(o32) || !aligned16(dO) || !aligned16(D) || !aligned16(dq_accum))
        return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    if ((rc = current_device(&status))) return rc;
    PreO32Args a{};
    a.o32 = o32;
    a.dO = dO;
    a.D = D;
    a.dq_accum = dq_accum;
    a.rows = static_cast<long long>(B) * H * N;
    a.d = d;
    return map_launch(launch_bwd_preprocess_o32(a, bf16, static_cast<cudaStream_t>(stream)));
}

int bwd_impl(const void* q, const void* k, const void* v, const void* dO, const float* lse,
             const float* D, float* dq_accum, void* dq, void* dk, void* dv, int B, int H, int Hkv,
             int N, int d, int causal, float scale, void* stream, bool bf16,
             const BwdOptions& opt = BwdOptions()) {
    const void* block_mask = opt.block_mask;
    const long long mask_stride = opt.mask_stride;
    float* dk32 = opt.dk32;
    float* dv32 = opt.dv32;
    const int acc32 = opt.acc32;
    const DropoutArgs* drop = opt.drop;
    const int splits = opt.splits;
    float* split_part = opt.split_part;
    // with fp32 gradient outputs (dk32, dv32) the 16-bit dk, dv are not used
    const bool f32 = dk32 != nullptr || dv32 != nullptr;
    if (f32 && (!dk32 || !dv32)) return ATTN_ERR_INVALID_ARG;
    if (f32 && !aligned16(dv32)) return ATTN_ERR_MISALIGNED;
    if (f32) dk = dv = dk32;
    // group split: shares in split_part, summed into the 16-bit dk, dv at the end
    if (splits < 1 || (splits > 1 && (f32 || !split_part || Hkv < 1 || H % Hkv != 0 ||
                                      (H / Hkv) % splits != 0)))
        return ATTN_ERR_INVALID_ARG;
    if (splits > 1 && !aligned16(split_part)) return ATTN_ERR_MISALIGNED;
    if (!q || !k || !v || !dO || !lse || !D || !dq_accum || !dq || !dk || !dv)
        return ATTN_ERR_INVALID_ARG;
    int rc = check_shape(B, H, N, d);
    if (rc) return rc;
    if ((rc = check_kv_heads(H, Hkv))) return rc;
    if ((rc = check_scale(scale))) return rc;
    if (block_mask != nullptr && (rc = check_sparse(block_mask, mask_stride, H, Hkv, N))) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
        !aligned16(D) || !aligned16(dq_accum) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
        return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    if ((rc = current_device(&status))) return rc;
    const int BH = B * H, BHkv = B * Hkv;
    CUtensorMap tq, tk, tv, tdo;
    if ((rc = make_map(&tq, q, BH, N, d, bf16)) || (rc = make_map(&tk, k, BHkv, N, d, bf16)) ||
        (rc = make_map(&tv, v, BHkv, N, d, bf16)) || (rc = make_map(&tdo, dO, BH, N, d, bf16)))
        return rc;
    CUtensorMap tdq, tdk, tdv;
    if ((rc = make_map_f32(&tdq, dq_accum, BH, N, d))) return rc;
    if (f32 || splits > 1) {
        tdk = tdv = tq;   // not used: the fp32 rows are written directly
    } else if ((rc = make_map(&tdk, dk, BHkv, N, d, bf16)) || (rc = make_map(&tdv, dv, BHkv, N, d, bf16))) {
        return rc;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    BwdArgs a{};
    a.lse = lse;
    a.D = D;
    a.dq_accum = dq_accum;
    a.dk = dk;
    a.dv = dv;
    a.status = status;
    a.N = N;
    a.BH = BH;
    a.H = H;
    a.Hkv = Hkv;
    a.BHkv = B * Hkv;
    a.num_kvblocks = (N + kTile - 1) / kTile;
    // the fp32 dQ rows and the Q, dO tiles of a head are re-read by each key-block CTA
    a.head_group = (Hkv == H) ? head_group_for(B * H, a.num_kvblocks, 8ll * N * d, kBwdGroupBytes) : 0;
    a.block_mask = static_cast<const uint8_t*>(block_mask);
    a.mask_head_stride = mask_stride;
    a.mask_cols = a.num_kvblocks;
    a.dk32 = dk32;
    a.dv32 = dv32;
    a.acc32 = acc32;
    if (drop != nullptr) a.drop = *drop;
    const long long kv_elems = static_cast<long long>(BHkv) * N * d;
    a.splits = splits;
    if (splits > 1) {
        a.dk32 = split_part;
        a.dv32 = split_part + splits * kv_elems;
        a.split_stride = kv_elems;
    }
    a.scale = scale;
    a.scale_log2 = scale * kLog2e;
    a.wait_polls = kDefaultWaitPolls;
    // one CTA per (batch, K / V head, key block): it loops over the head's group
    if ((rc = map_launch(launch_bwd(tq, tk, tv, tdo, tdq, tdk, tdv, a, BHkv, d, causal != 0, bf16, st))))
        return rc;
    DqConvertArgs c{};
    c.dq_accum = dq_accum;
    c.dq = dq;
    c.elems = static_cast<long long>(BH) * N * d;
    c.scale = scale;
    if ((rc = map_launch(launch_dq_convert(c, bf16, st)))) return rc;
    if (splits > 1) {
        SplitSumArgs sk{a.dk32, dk, kv_elems, splits}, sv{a.dv32, dv, kv_elems, splits};
        if ((rc = map_launch(launch_split_sum(sk, bf16, st)))) return rc;
        if ((rc = map_launch(launch_split_sum(sv, bf16, st)))) return rc;
    }
    return ATTN_OK;
}

// Tensor maps over a packed variable-length [total, Hh, d] array (the valid
// tokens of all sequences concatenated, heads interleaved): dimensions
// (d, token, head) with strides (Hh * d, d) elements, so the kernels address it
// with the same (column, row, head) coordinates as a dense [BH, N, d] array.
int make_map_packed(CUtensorMap* m, const void* base, int total, int Hh, int d, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return ATTN_ERR_LAUNCH;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(total),
                                static_cast<cuuint64_t>(Hh)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Hh) * d * 2, static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBoxCols), static_cast<cuuint32_t>(kTile), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

// Tile map over a packed [total, Hh, d] 16-bit array (rows = tokens).
int make_tile_map_packed(CUtensorMap* m, const void* base, int total, int Hh, int d, bool bf16) {
    return encode_tile_map(m, base, static_cast<cuuint64_t>(total), static_cast<cuuint64_t>(Hh), d,
                           static_cast<cuuint64_t>(Hh) * d * 2, static_cast<cuuint64_t>(d) * 2, bf16);
}

int make_map_packed_f32(CUtensorMap* m, const void* base, int total, int Hh, int d) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return ATTN_ERR_LAUNCH;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(total),
                                static_cast<cuuint64_t>(Hh)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Hh) * d * 4, static_cast<cuuint64_t>(d) * 4};
    const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(kTile), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

int check_varlen(const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv, int d) {
    if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || total < 0 || max_seqlen < 1 || max_seqlen > (1 << 24)) return ATTN_ERR_INVALID_ARG;
    if (H < 1 || static_cast<long long>(total) * H > 2147483647LL) return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H > 2147483647LL) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEAD_DIM;
    return check_kv_heads(H, Hkv);
}

// Keys of their own lengths (cu_seqlens_k != nullptr): sequence b's keys are
// rows [cu_seqlens_k[b], cu_seqlens_k[b+1]) of the [total_k, Hkv, d] K and V.
struct VarlenKeys {
    const int* cu_seqlens_k = nullptr;
    int total_k = 0;
    int max_seqlen_k = 0;
};

int check_varlen_keys(const VarlenKeys& kv, int Hkv) {
    if (kv.cu_seqlens_k == nullptr) return ATTN_OK;
    if (reinterpret_cast<uintptr_t>(kv.cu_seqlens_k) & 3u) return ATTN_ERR_INVALID_ARG;
    if (kv.total_k < 0 || kv.max_seqlen_k < 1 || kv.max_seqlen_k > (1 << 24)) return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(kv.total_k) * Hkv > 2147483647LL) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

int fwd_varlen_impl(const void* q, const void* k, const void* v, void* o, float* o32, float* lse,
                    const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv, int d,
                    int causal, float scale, void* stream, bool bf16, VarlenKeys kv = {}) {
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
    int rc = check_varlen(cu_seqlens, B, total, max_seqlen, H, Hkv, d);
    if (rc) return rc;
    if ((rc = check_varlen_keys(kv, Hkv))) return rc;
    const bool own_keys = kv.cu_seqlens_k != nullptr;
    const int total_k = own_keys ? kv.total_k : total;
    if ((rc = check_scale(scale))) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        (o32 != nullptr && !aligned16(o32)))
        return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    if ((rc = current_device(&status))) return rc;
    if (total == 0) return ATTN_OK;   // no query tokens: nothing to compute
    CUtensorMap tq, tk, tv, to, to32;
    if ((rc = make_tile_map_packed(&tq, q, total, H, d, bf16)) || (rc = make_map_packed(&to, o, total, H, d, bf16)))
        return rc;
    if (total_k > 0) {
        if ((rc = make_tile_map_packed(&tk, k, total_k, Hkv, d, bf16)) ||
            (rc = make_tile_map_packed(&tv, v, total_k, Hkv, d, bf16)))
            return rc;
    } else {
        tk = tq;   // no key rows at all: every CTA writes empty rows and loads nothing
        tv = tq;
    }
    if (o32 != nullptr) {
        if ((rc = make_map_packed_f32(&to32, o32, total, H, d))) return rc;
    } else {
        to32 = to;
    }
    FwdArgs a{};
    a.o = o;
    a.o32 = o32;
    a.lse = lse;
    a.status = status;
    a.N = max_seqlen;
    a.BH = B * H;
    a.H = H;
    a.Hkv = Hkv;
    a.num_qblocks = (max_seqlen + 2 * kTile - 1) / (2 * kTile);
    a.cu_seqlens = cu_seqlens;
    a.total = total;
    a.max_seqlen = max_seqlen;
    a.cu_seqlens_k = kv.cu_seqlens_k;
    a.total_k = total_k;
    a.max_seqlen_k = own_keys ? kv.max_seqlen_k : max_seqlen;
    a.scale_log2 = scale * kLog2e;
    a.wait_polls = kDefaultWaitPolls;
    return map_launch(launch_fwd(tq, tk, tv, to, to32, a, B * H, d, causal != 0, bf16,
                                 static_cast<cudaStream_t>(stream)));
}

int pre_o32_varlen_impl(const float* o32, const void* dO, float* D, float* dq_accum, int total,
                        int H, int d, void* stream, bool bf16) {
    if (!o32 || !dO || !D || !dq_accum) return ATTN_ERR_INVALID_ARG;
    if (total < 0 || H < 1 || static_cast<long long>(total) * H > 2147483647LL) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEAD_DIM;
    if (!aligned16(o32) || !aligned16(dO) || !aligned16(D) || !aligned16(dq_accum))
        return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    int rc = current_device(&status);
    if (rc) return rc;
    if (total == 0) return ATTN_OK;
    // the packed [total, H, d] rows, one D value per row: D is [total, H]
    PreO32Args a{};
    a.o32 = o32;
    a.dO = dO;
    a.D = D;
    a.dq_accum = dq_accum;
    a.rows = static_cast<long long>(total) * H;
    a.d = d;
    return map_launch(launch_bwd_preprocess_o32(a, bf16, static_cast<cudaStream_t>(stream)));
}

int bwd_varlen_impl(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                    const float* D, float* dq_accum, void* dq, void* dk, void* dv,
                    const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv, int d,
                    int causal, float scale, void* stream, bool bf16, VarlenKeys kv = {}) {
    if (!q || !k || !v || !dO || !lse || !D || !dq_accum || !dq || !dk || !dv)
        return ATTN_ERR_INVALID_ARG;
    int rc = check_varlen(cu_seqlens, B, total, max_seqlen, H, Hkv, d);
    if (rc) return rc;
    if ((rc = check_varlen_keys(kv, Hkv))) return rc;
    const bool own_keys = kv.cu_seqlens_k != nullptr;
    const int total_k = own_keys ? kv.total_k : total;
    const int max_seqlen_k = own_keys ? kv.max_seqlen_k : max_seqlen;
    if ((rc = check_scale(scale))) return rc;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
        !aligned16(D) || !aligned16(dq_accum) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
        return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    if ((rc = current_device(&status))) return rc;
    if (total == 0 && total_k == 0) return ATTN_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DqConvertArgs c{};
    c.dq_accum = dq_accum;
    c.dq = dq;
    c.elems = static_cast<long long>(total) * H * d;
    c.scale = scale;
    // no key rows: dK, dV are empty and every dQ row is 0 (dq_accum was zeroed)
    if (total_k == 0) return map_launch(launch_dq_convert(c, bf16, st));
    CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
    if ((rc = make_map_packed(&tk, k, total_k, Hkv, d, bf16)) || (rc = make_map_packed(&tv, v, total_k, Hkv, d, bf16)) ||
        (rc = make_map_packed(&tdk, dk, total_k, Hkv, d, bf16)) || (rc = make_map_packed(&tdv, dv, total_k, Hkv, d, bf16)))
        return rc;
    if (total > 0) {
        if ((rc = make_map_packed(&tq, q, total, H, d, bf16)) || (rc = make_map_packed(&tdo, dO, total, H, d, bf16)) ||
            (rc = make_map_packed_f32(&tdq, dq_accum, total, H, d)))
            return rc;
    } else {
        tq = tk;   // no query rows: every CTA writes dK = dV = 0 and loads no query
        tdo = tk;
        tdq = tk;
    }
    BwdArgs a{};
    a.lse = lse;
    a.D = D;
    a.dq_accum = dq_accum;
    a.dk = dk;
    a.dv = dv;
    a.status = status;
    a.N = max_seqlen;
    a.BH = B * H;
    a.H = H;
    a.Hkv = Hkv;
    a.BHkv = B * Hkv;
    a.num_kvblocks = (max_seqlen_k + kTile - 1) / kTile;
    a.cu_seqlens = cu_seqlens;
    a.total = total;
    a.max_seqlen = max_seqlen;
    a.cu_seqlens_k = kv.cu_seqlens_k;
    a.total_k = total_k;
    a.max_seqlen_k = max_seqlen_k;
    a.scale = scale;
    a.scale_log2 = scale * kLog2e;
    a.wait_polls = kDefaultWaitPolls;
    // one CTA per (sequence, K / V head, key block); blocks past a sequence exit
    if ((rc = map_launch(launch_bwd(tq, tk, tv, tdo, tdq, tdk, tdv, a, B * Hkv, d, causal != 0, bf16, st))))
        return rc;
    if (total == 0) return ATTN_OK;
    return map_launch(launch_dq_convert(c, bf16, st));
}

__global__ void selftest_timeout_kernel(int* status, unsigned int max_polls) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;
    const uint32_t b = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Nothing ever arrives on the barrier: the wait must run out and report.
    const WaitCtx wc{&abort_flag, status, max_polls};
    if (threadIdx.x == 0) (void)wait_bar(wc, b, 0);
}

int merge_impl(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
               void* o_out, long long rows, int d, void* stream, bool bf16) {
    if (!o_acc || !lse_acc || !o_part || !lse_part || rows < 0) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED_HEAD_DIM;
    if (!aligned16(o_acc) || !aligned16(o_part) || (o_out && !aligned16(o_out)))
        return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    int rc = current_device(&status);
    if (rc) return rc;
    if (rows == 0) return ATTN_OK;
    MergeArgs a{o_acc, lse_acc, o_part, lse_part, o_out, rows, d};
    return map_launch(launch_merge(a, bf16, static_cast<cudaStream_t>(stream)));
}

int convert_impl(const float* x, void* y, long long elems, float scale, void* stream, bool bf16) {
    if (!x || !y || elems < 0 || elems % 8 != 0 || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return ATTN_ERR_MISALIGNED;
    int* status = nullptr;
    int rc = current_device(&status);
    if (rc) return rc;
    if (elems == 0) return ATTN_OK;
    DqConvertArgs c{};
    c.dq_accum = x;
    c.dq = y;
    c.elems = elems;
    c.scale = scale;
    return map_launch(launch_dq_convert(c, bf16, static_cast<cudaStream_t>(stream)));
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, int causal, float scale, void* stream) {
    return fwd_impl(q, k, v, o, nullptr, lse, B, H, H, N, d, causal, scale, stream, true);
}

int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, int causal, float scale, void* stream) {
    return fwd_impl(q, k, v, o, nullptr, lse, B, H, H, N, d, causal, scale, stream, false);
}

int attn_fwd_train(const void* q, const void* k, const void* v, void* o, float* o32, float* lse,
                   int B, int H, int N, int d, int causal, float scale, void* stream) {
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, o32, lse, B, H, H, N, d, causal, scale, stream, true);
}

int attn_fwd_train_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                       float* lse, int B, int H, int N, int d, int causal, float scale,
                       void* stream) {
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, o32, lse, B, H, H, N, d, causal, scale, stream, false);
}

int attn_bwd_preprocess_o32(const float* o32, const void* dO, float* D, float* dq_accum, int B,
                            int H, int N, int d, void* stream) {
    return pre_o32_impl(o32, dO, D, dq_accum, B, H, N, d, stream, true);
}

int attn_bwd_preprocess_o32_f16(const float* o32, const void* dO, float* D, float* dq_accum,
                                int B, int H, int N, int d, void* stream) {
    return pre_o32_impl(o32, dO, D, dq_accum, B, H, N, d, stream, false);
}

int attn_bwd_preprocess(const void* q, const void* k, const void* v, const void* dO,
                        const float* lse, float* D, float* dq_accum, int B, int H, int N, int d,
                        int causal, float scale, void* stream) {
    return pre_impl(q, k, v, dO, lse, D, dq_accum, B, H, H, N, d, causal, scale, stream, true);
}

int attn_bwd_preprocess_f16(const void* q, const void* k, const void* v, const void* dO,
                            const float* lse, float* D, float* dq_accum, int B, int H, int N,
                            int d, int causal, float scale, void* stream) {
    return pre_impl(q, k, v, dO, lse, D, dq_accum, B, H, H, N, d, causal, scale, stream, false);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* dO, const float* lse,
             const float* D, float* dq_accum, void* dq, void* dk, void* dv, int B, int H, int N,
             int d, int causal, float scale, void* stream) {
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, H, N, d, causal, scale, stream,
                    true);
}

int attn_bwd_f16(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                 const float* D, float* dq_accum, void* dq, void* dk, void* dv, int B, int H,
                 int N, int d, int causal, float scale, void* stream) {
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, H, N, d, causal, scale, stream,
                    false);
}

int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Hkv, int N, int d, int causal, float scale, void* stream) {
    return fwd_impl(q, k, v, o, nullptr, lse, B, H, Hkv, N, d, causal, scale, stream, true);
}

int attn_fwd_gqa_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int Hkv, int N, int d, int causal, float scale, void* stream) {
    return fwd_impl(q, k, v, o, nullptr, lse, B, H, Hkv, N, d, causal, scale, stream, false);
}

int attn_fwd_train_gqa(const void* q, const void* k, const void* v, void* o, float* o32,
                       float* lse, int B, int H, int Hkv, int N, int d, int causal, float scale,
                       void* stream) {
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, o32, lse, B, H, Hkv, N, d, causal, scale, stream, true);
}

int attn_fwd_train_gqa_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                           float* lse, int B, int H, int Hkv, int N, int d, int causal,
                           float scale, void* stream) {
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, o32, lse, B, H, Hkv, N, d, causal, scale, stream, false);
}

int attn_bwd_preprocess_gqa(const void* q, const void* k, const void* v, const void* dO,
                            const float* lse, float* D, float* dq_accum, int B, int H, int Hkv,
                            int N, int d, int causal, float scale, void* stream) {
    return pre_impl(q, k, v, dO, lse, D, dq_accum, B, H, Hkv, N, d, causal, scale, stream, true);
}

int attn_bwd_preprocess_gqa_f16(const void* q, const void* k, const void* v, const void* dO,
                                const float* lse, float* D, float* dq_accum, int B, int H,
                                int Hkv, int N, int d, int causal, float scale, void* stream) {
    return pre_impl(q, k, v, dO, lse, D, dq_accum, B, H, Hkv, N, d, causal, scale, stream, false);
}

int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                 const float* D, float* dq_accum, void* dq, void* dk, void* dv, int B, int H,
                 int Hkv, int N, int d, int causal, float scale, void* stream) {
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, Hkv, N, d, causal, scale,
                    stream, true);
}

int attn_bwd_gqa_f16(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                     void* dv, int B, int H, int Hkv, int N, int d, int causal, float scale,
                     void* stream) {
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, Hkv, N, d, causal, scale,
                    stream, false);
}

int attn_fwd_bsparse(const void* q, const void* k, const void* v, void* o, float* lse,
                     const void* block_mask, long long mask_head_stride, int B, int H, int N,
                     int d, int causal, float scale, void* stream) {
    if (!block_mask) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, nullptr, lse, B, H, H, N, d, causal, scale, stream, true,
                    sparse_fwd(block_mask, mask_head_stride));
}

int attn_fwd_bsparse_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                         const void* block_mask, long long mask_head_stride, int B, int H, int N,
                         int d, int causal, float scale, void* stream) {
    if (!block_mask) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, nullptr, lse, B, H, H, N, d, causal, scale, stream, false,
                    sparse_fwd(block_mask, mask_head_stride));
}

int attn_fwd_train_bsparse(const void* q, const void* k, const void* v, void* o, float* o32,
                           float* lse, const void* block_mask, long long mask_head_stride, int B,
                           int H, int N, int d, int causal, float scale, void* stream) {
    if (!block_mask) return ATTN_ERR_INVALID_ARG;
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, o32, lse, B, H, H, N, d, causal, scale, stream, true,
                    sparse_fwd(block_mask, mask_head_stride));
}

int attn_fwd_train_bsparse_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                               float* lse, const void* block_mask, long long mask_head_stride,
                               int B, int H, int N, int d, int causal, float scale, void* stream) {
    if (!block_mask) return ATTN_ERR_INVALID_ARG;
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, o32, lse, B, H, H, N, d, causal, scale, stream, false,
                    sparse_fwd(block_mask, mask_head_stride));
}

int attn_bwd_bsparse(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                     void* dv, const void* block_mask, long long mask_head_stride, int B, int H,
                     int N, int d, int causal, float scale, void* stream) {
    if (!block_mask) return ATTN_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, H, N, d, causal, scale,
                    stream, true, sparse_bwd(block_mask, mask_head_stride));
}

int attn_bwd_bsparse_f16(const void* q, const void* k, const void* v, const void* dO,
                         const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                         void* dv, const void* block_mask, long long mask_head_stride, int B,
                         int H, int N, int d, int causal, float scale, void* stream) {
    if (!block_mask) return ATTN_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, H, N, d, causal, scale,
                    stream, false, sparse_bwd(block_mask, mask_head_stride));
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv,
                    int d, int causal, float scale, void* stream) {
    return fwd_varlen_impl(q, k, v, o, nullptr, lse, cu_seqlens, B, total, max_seqlen, H, Hkv, d,
                           causal, scale, stream, true);
}

int attn_fwd_varlen_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv,
                        int d, int causal, float scale, void* stream) {
    return fwd_varlen_impl(q, k, v, o, nullptr, lse, cu_seqlens, B, total, max_seqlen, H, Hkv, d,
                           causal, scale, stream, false);
}

int attn_fwd_train_varlen(const void* q, const void* k, const void* v, void* o, float* o32,
                          float* lse, const int* cu_seqlens, int B, int total, int max_seqlen,
                          int H, int Hkv, int d, int causal, float scale, void* stream) {
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return fwd_varlen_impl(q, k, v, o, o32, lse, cu_seqlens, B, total, max_seqlen, H, Hkv, d,
                           causal, scale, stream, true);
}

int attn_fwd_train_varlen_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                              float* lse, const int* cu_seqlens, int B, int total, int max_seqlen,
                              int H, int Hkv, int d, int causal, float scale, void* stream) {
    if (!o32) return ATTN_ERR_INVALID_ARG;
    return fwd_varlen_impl(q, k, v, o, o32, lse, cu_seqlens, B, total, max_seqlen, H, Hkv, d,
                           causal, scale, stream, false);
}

int attn_bwd_preprocess_o32_varlen(const float* o32, const void* dO, float* D, float* dq_accum,
                                   int total, int H, int d, void* stream) {
    return pre_o32_varlen_impl(o32, dO, D, dq_accum, total, H, d, stream, true);
}

int attn_bwd_preprocess_o32_varlen_f16(const float* o32, const void* dO, float* D,
                                       float* dq_accum, int total, int H, int d, void* stream) {
    return pre_o32_varlen_impl(o32, dO, D, dq_accum, total, H, d, stream, false);
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                    const float* D, float* dq_accum, void* dq, void* dk, void* dv,
                    const int* cu_seqlens, int B, int total, int max_seqlen, int H, int Hkv, int d,
                    int causal, float scale, void* stream) {
    return bwd_varlen_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, cu_seqlens, B, total,
                           max_seqlen, H, Hkv, d, causal, scale, stream, true);
}

int attn_bwd_varlen_f16(const void* q, const void* k, const void* v, const void* dO,
                        const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                        void* dv, const int* cu_seqlens, int B, int total, int max_seqlen, int H,
                        int Hkv, int d, int causal, float scale, void* stream) {
    return bwd_varlen_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, cu_seqlens, B, total,
                           max_seqlen, H, Hkv, d, causal, scale, stream, false);
}

int attn_fwd_varlen_qk(const void* q, const void* k, const void* v, void* o, float* lse,
                       const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int total_q,
                       int total_k, int max_seqlen_q, int max_seqlen_k, int H, int Hkv, int d,
                       int causal, float scale, void* stream) {
    if (!cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    return fwd_varlen_impl(q, k, v, o, nullptr, lse, cu_seqlens_q, B, total_q, max_seqlen_q, H, Hkv,
                           d, causal, scale, stream, true, {cu_seqlens_k, total_k, max_seqlen_k});
}

int attn_fwd_varlen_qk_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                           const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int total_q,
                           int total_k, int max_seqlen_q, int max_seqlen_k, int H, int Hkv, int d,
                           int causal, float scale, void* stream) {
    if (!cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    return fwd_varlen_impl(q, k, v, o, nullptr, lse, cu_seqlens_q, B, total_q, max_seqlen_q, H, Hkv,
                           d, causal, scale, stream, false, {cu_seqlens_k, total_k, max_seqlen_k});
}

int attn_fwd_train_varlen_qk(const void* q, const void* k, const void* v, void* o, float* o32,
                             float* lse, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                             int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H,
                             int Hkv, int d, int causal, float scale, void* stream) {
    if (!o32 || !cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    return fwd_varlen_impl(q, k, v, o, o32, lse, cu_seqlens_q, B, total_q, max_seqlen_q, H, Hkv, d,
                           causal, scale, stream, true, {cu_seqlens_k, total_k, max_seqlen_k});
}

int attn_fwd_train_varlen_qk_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                                 float* lse, const int* cu_seqlens_q, const int* cu_seqlens_k,
                                 int B, int total_q, int total_k, int max_seqlen_q,
                                 int max_seqlen_k, int H, int Hkv, int d, int causal, float scale,
                                 void* stream) {
    if (!o32 || !cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    return fwd_varlen_impl(q, k, v, o, o32, lse, cu_seqlens_q, B, total_q, max_seqlen_q, H, Hkv, d,
                           causal, scale, stream, false, {cu_seqlens_k, total_k, max_seqlen_k});
}

int attn_bwd_varlen_qk(const void* q, const void* k, const void* v, const void* dO,
                       const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                       void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                       int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H,
                       int Hkv, int d, int causal, float scale, void* stream) {
    if (!cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    return bwd_varlen_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, cu_seqlens_q, B, total_q,
                           max_seqlen_q, H, Hkv, d, causal, scale, stream, true,
                           {cu_seqlens_k, total_k, max_seqlen_k});
}

int attn_bwd_varlen_qk_f16(const void* q, const void* k, const void* v, const void* dO,
                           const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                           void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B,
                           int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H,
                           int Hkv, int d, int causal, float scale, void* stream) {
    if (!cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    return bwd_varlen_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, cu_seqlens_q, B, total_q,
                           max_seqlen_q, H, Hkv, d, causal, scale, stream, false,
                           {cu_seqlens_k, total_k, max_seqlen_k});
}

const char* attn_status_string(int s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED_HEAD_DIM: return "unsupported head dimension (d must be 64 or 128)";
        case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case ATTN_ERR_UNSUPPORTED_DEVICE: return "current device is not an sm_103 GPU";
        case ATTN_ERR_LAUNCH: return "CUDA launch failed";
        case ATTN_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
        case ATTN_ERR_DEVICE_FAULT: return "CUDA reported an error while synchronising";
        case ATTN_ERR_SCRATCH_TOO_SMALL: return "problem too large for the fixed no-allocation scratch array";
        default: return "unknown status";
    }
}

int attn_get_device_status(void* stream) {
    int* status = nullptr;
    int rc = current_device(&status);
    if (rc) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_DEVICE_FAULT;
    }
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_DEVICE_FAULT;
    }
    if (v == DEV_OK) return ATTN_OK;
    return v == DEV_TIMEOUT ? ATTN_ERR_TIMEOUT : ATTN_ERR_LAUNCH;
}

int attn_selftest_timeout(int timeout_us, void* stream) {
    if (timeout_us < 1 || timeout_us > 1000000) return ATTN_ERR_INVALID_ARG;
    int* status = nullptr;
    int rc = current_device(&status);
    if (rc) return rc;
    selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        status, static_cast<unsigned int>((timeout_us + 1) / 2));   // about 2 us per poll
    return map_launch(cudaGetLastError());
}

const char* attn_version(void) { return "io_aware_exact_gb300 0.1 (sm_103a)"; }

int attn_merge(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
               void* o_out, long long rows, int d, void* stream) {
    return attn::merge_impl(o_acc, lse_acc, o_part, lse_part, o_out, rows, d, stream, true);
}

int attn_merge_f16(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                   void* o_out, long long rows, int d, void* stream) {
    return attn::merge_impl(o_acc, lse_acc, o_part, lse_part, o_out, rows, d, stream, false);
}

int attn_bwd_acc(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                 const float* D, float* dq_accum, void* dq, float* dk32, float* dv32,
                 int accumulate, int B, int H, int Hkv, int N, int d, int causal, float scale,
                 void* stream) {
    if (!dk32 || !dv32) return ATTN_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, nullptr, nullptr, B, H, Hkv, N, d, causal,
                    scale, stream, true, f32_bwd(dk32, dv32, accumulate != 0));
}

int attn_bwd_acc_f16(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, float* dq_accum, void* dq, float* dk32,
                     float* dv32, int accumulate, int B, int H, int Hkv, int N, int d,
                     int causal, float scale, void* stream) {
    if (!dk32 || !dv32) return ATTN_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, nullptr, nullptr, B, H, Hkv, N, d, causal,
                    scale, stream, false, f32_bwd(dk32, dv32, accumulate != 0));
}

int attn_fwd_train_dropout(const void* q, const void* k, const void* v, void* o, float* o32,
                           float* lse, float p_drop, unsigned long long seed, unsigned int offset,
                           int B, int H, int N, int d, int causal, float scale, void* stream) {
    DropoutArgs dr{};
    int rc = make_dropout(p_drop, seed, offset, &dr);
    if (rc) return rc;
    if (!o32) return ATTN_ERR_INVALID_ARG;
    FwdOptions opt;
    opt.drop = &dr;
    return fwd_impl(q, k, v, o, o32, lse, B, H, H, N, d, causal, scale, stream, true, opt);
}

int attn_fwd_train_dropout_f16(const void* q, const void* k, const void* v, void* o, float* o32,
                               float* lse, float p_drop, unsigned long long seed,
                               unsigned int offset, int B, int H, int N, int d, int causal,
                               float scale, void* stream) {
    DropoutArgs dr{};
    int rc = make_dropout(p_drop, seed, offset, &dr);
    if (rc) return rc;
    if (!o32) return ATTN_ERR_INVALID_ARG;
    FwdOptions opt;
    opt.drop = &dr;
    return fwd_impl(q, k, v, o, o32, lse, B, H, H, N, d, causal, scale, stream, false, opt);
}

int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                     void* dv, float p_drop, unsigned long long seed, unsigned int offset, int B,
                     int H, int N, int d, int causal, float scale, void* stream) {
    DropoutArgs dr{};
    int rc = make_dropout(p_drop, seed, offset, &dr);
    if (rc) return rc;
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, H, N, d, causal, scale,
                    stream, true, drop_bwd(&dr));
}

int attn_bwd_dropout_f16(const void* q, const void* k, const void* v, const void* dO,
                         const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                         void* dv, float p_drop, unsigned long long seed, unsigned int offset,
                         int B, int H, int N, int d, int causal, float scale, void* stream) {
    DropoutArgs dr{};
    int rc = make_dropout(p_drop, seed, offset, &dr);
    if (rc) return rc;
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, H, N, d, causal, scale,
                    stream, false, drop_bwd(&dr));
}

int attn_gqa_split_hint(int B, int H, int Hkv, int N, int causal) {
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || N < 1) return 1;
    const int G = H / Hkv;
    const double nb = static_cast<double>((N + kTile - 1) / kTile);
    // query-block iterations of the whole launch and of the heaviest CTA
    const double total = static_cast<double>(B) * H * (causal ? nb * (nb + 1) / 2 : nb * nb);
    const double per_sm = total / device_sm_count();
    for (int s = 1; s <= G; ++s)
        if (G % s == 0 && (G / s) * nb <= per_sm) return s;
    return G;
}

int attn_bwd_gqa_split(const void* q, const void* k, const void* v, const void* dO,
                       const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                       void* dv, float* dkv_part, int splits, int B, int H, int Hkv, int N,
                       int d, int causal, float scale, void* stream) {
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, Hkv, N, d, causal, scale,
                    stream, true, split_bwd(splits, dkv_part));
}

int attn_bwd_gqa_split_f16(const void* q, const void* k, const void* v, const void* dO,
                           const float* lse, const float* D, float* dq_accum, void* dq, void* dk,
                           void* dv, float* dkv_part, int splits, int B, int H, int Hkv, int N,
                           int d, int causal, float scale, void* stream) {
    return bwd_impl(q, k, v, dO, lse, D, dq_accum, dq, dk, dv, B, H, Hkv, N, d, causal, scale,
                    stream, false, split_bwd(splits, dkv_part));
}

int attn_convert(const float* x, void* y, long long elems, float scale, void* stream) {
    return attn::convert_impl(x, y, elems, scale, stream, true);
}

int attn_convert_f16(const float* x, void* y, long long elems, float scale, void* stream) {
    return attn::convert_impl(x, y, elems, scale, stream, false);
}

}  // extern "C"
