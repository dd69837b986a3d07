// moe_io.cu -- the steps on either side of the grouped GEMM in an MoE layer.
//
// 1. hg_quantize_gather_acts: BF16 token activations -> FP8 E4M3 codes with
//    one E8M0 scale per 128-K group, written directly in the plan's sorted
//    row order (row r takes token sorted_to_src[r] / top_k).  The scale rule
//    is the one the workloads state: scale = 2^e with e the smallest integer
//    such that amax <= 448 * 2^e (amax = 0 gives e = 0), e clamped to
//    [-127, 127]; codes are E4M3 round-to-nearest-even of x / scale.  The
//    rowwise MXFP8 cast of TransformerEngine PR #3459 ("non-TMA MXFP8
//    cast-only kernels", description) is the same kind of register-only,
//    HBM-bound cast, with 32-element blocks there and 128 here.
//    hg_quantize_scatter_acts: the same codes, each token quantised once and
//    stored to its top_k sorted rows src_to_sorted[t*k + j] (the plan's
//    inverse permutation): the token is read once instead of top_k times.
// 2. hg_combine_topk: out[t, :] = sum_j w[t, j] * y[src_to_sorted[t*k+j], :]
//    in FP32, j ascending, rounded once to BF16; terms whose id was dropped
//    by the plan (src_to_sorted = -1) are skipped.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "hg_internal.cuh"

namespace hg {
namespace {

constexpr int kGroup = 128;

// Smallest e with amax <= 448 * 2^e, from the bits of amax (exact, no
// floating-point division or logarithm).  amax = f * 2^p with f in [1, 2):
// amax <= 1.75 * 2^(8+e)  <=>  e >= p - 8 when f <= 1.75, else e >= p - 7.
__device__ __forceinline__ int scale_exponent(float amax) {
    if (amax == 0.0f) return 0;
    const uint32_t bits = __float_as_uint(amax);
    int p;
    uint32_t mant;
    const uint32_t be = (bits >> 23) & 0xFFu;
    if (be == 0) {                         // subnormal: normalise
        const uint32_t m = bits & 0x7FFFFFu;
        const int lz = __clz(m) - 8;       // shift that brings the leading 1 to bit 23
        p = -126 - lz;
        mant = (m << lz) & 0x7FFFFFu;
    } else {
        p = static_cast<int>(be) - 127;
        mant = bits & 0x7FFFFFu;
    }
    int e = p - 8 + (mant > 0x600000u ? 1 : 0);
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// One 256-thread block per sorted row and iteration: the row's source index is
// read once, then each half-warp takes groups hw, hw+16, hw+32, ... of the row
// with all its 16-byte loads issued before any is used (lane j of the half
// holds elements 8j .. 8j+7 of a group).
constexpr int kQThreads = 256;
constexpr int kQHalves = kQThreads / 16;
constexpr int kQMaxIter = 4;                       // groups per half-warp held in registers

struct GroupCodes {
    uint32_t lo, hi;        // this lane's 8 E4M3 codes
    uint8_t scale;          // the group's E8M0 code
};

// Lane j of a half-warp holds elements 8j .. 8j+7 of one 128-element group;
// every lane of the warp must call this (the amax reduction shuffles).
__device__ __forceinline__ GroupCodes quantize_codes(const uint4 v) {
    float f[8];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = 0.0f;
    bool nonfinite = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        amax = fmaxf(amax, fabsf(f[i]));
        nonfinite |= !isfinite(f[i]);
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        nonfinite |= __shfl_xor_sync(0xFFFFFFFFu, nonfinite ? 1 : 0, o) != 0;
    }
    GroupCodes c;
    if (nonfinite) {
        c.scale = 0xFF;                            // E8M0 NaN
        c.lo = c.hi = 0x7F7F7F7Fu;                 // E4M3 NaN
    } else {
        const int e = scale_exponent(amax);
        c.scale = static_cast<uint8_t>(127 + e);
        // 2^-e from its bits: finite BF16 inputs give e <= 120, so the
        // biased exponent 127 - e stays in [7, 254] (a normal float).
        const float inv = __int_as_float((127 - e) << 23);
        uint32_t b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            b[i] = __nv_cvt_float_to_fp8(f[i] * inv, __NV_SATFINITE, __NV_E4M3);
        }
        c.lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
        c.hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    }
    return c;
}

__device__ __forceinline__ void quantize_group(const uint4 v, uint8_t* dst, uint8_t* scale_dst,
                                               int j) {
    const GroupCodes c = quantize_codes(v);
    if (dst == nullptr) return;
    *reinterpret_cast<uint2*>(dst + 8 * j) = make_uint2(c.lo, c.hi);
    if (j == 0) *scale_dst = c.scale;
}

__global__ void __launch_bounds__(kQThreads)
quantize_gather_kernel(const uint16_t* __restrict__ x, int K, int top_k,
                       const int32_t* __restrict__ sorted_to_src, int rows,
                       uint8_t* __restrict__ a_fp8, uint8_t* __restrict__ a_scale) {
    const int G = K / kGroup;
    const int hw = threadIdx.x >> 4;
    const int j = threadIdx.x & 15;
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const int src = __ldg(sorted_to_src + r);
        if (src < 0) continue;                              // uniform across the block
        const uint16_t* xrow = x + static_cast<long long>(src / top_k) * K;
        uint8_t* arow = a_fp8 + static_cast<long long>(r) * K;
        uint8_t* srow = a_scale + static_cast<long long>(r) * G;
        for (int g0 = 0; g0 < G; g0 += kQHalves * kQMaxIter) {
            uint4 v[kQMaxIter];
#pragma unroll
            for (int k = 0; k < kQMaxIter; ++k) {
                const int g = g0 + hw + kQHalves * k;
                v[k] = make_uint4(0, 0, 0, 0);
                if (g < G) v[k] = __ldg(reinterpret_cast<const uint4*>(xrow + g * kGroup) + j);
            }
#pragma unroll
            for (int k = 0; k < kQMaxIter; ++k) {
                const int g = g0 + hw + kQHalves * k;
                // every lane takes part in the half-warp reductions; only
                // lanes of a real group write
                quantize_group(v[k], g < G ? arow + g * kGroup : nullptr, srow + g, j);
            }
        }
    }
}

// One 256-thread block per token and pass: the token's destination rows are
// read into shared memory, its groups are loaded and quantised once (as in
// quantize_gather_kernel), and each half-warp stores its group's codes and
// scale to every destination row in [0, rows).
constexpr int kMaxScatterTopK = 64;

__global__ void __launch_bounds__(kQThreads)
quantize_scatter_kernel(const uint16_t* __restrict__ x, int M, int K, int top_k,
                        const int32_t* __restrict__ src_to_sorted, int rows,
                        uint8_t* __restrict__ a_fp8, uint8_t* __restrict__ a_scale) {
    __shared__ int s_dst[kMaxScatterTopK];
    const int G = K / kGroup;
    const int hw = threadIdx.x >> 4;
    const int j = threadIdx.x & 15;
    for (int t = blockIdx.x; t < M; t += gridDim.x) {
        if (threadIdx.x < top_k) {
            const int r = __ldg(src_to_sorted + static_cast<long long>(t) * top_k + threadIdx.x);
            s_dst[threadIdx.x] = (r >= 0 && r < rows) ? r : -1;
        }
        __syncthreads();
        const uint16_t* xrow = x + static_cast<long long>(t) * K;
        for (int g0 = 0; g0 < G; g0 += kQHalves * kQMaxIter) {
            uint4 v[kQMaxIter];
#pragma unroll
            for (int k = 0; k < kQMaxIter; ++k) {
                const int g = g0 + hw + kQHalves * k;
                v[k] = make_uint4(0, 0, 0, 0);
                if (g < G) v[k] = __ldg(reinterpret_cast<const uint4*>(xrow + g * kGroup) + j);
            }
#pragma unroll
            for (int k = 0; k < kQMaxIter; ++k) {
                const int g = g0 + hw + kQHalves * k;
                const GroupCodes c = quantize_codes(v[k]);   // every lane: shuffles inside
                if (g < G) {
                    for (int d = 0; d < top_k; ++d) {
                        const int r = s_dst[d];
                        if (r < 0) continue;
                        *reinterpret_cast<uint2*>(a_fp8 + static_cast<long long>(r) * K +
                                                  g * kGroup + 8 * j) = make_uint2(c.lo, c.hi);
                        if (j == 0) a_scale[static_cast<long long>(r) * G + g] = c.scale;
                    }
                }
            }
        }
        __syncthreads();   // s_dst is rewritten for the next token
    }
}

// Work item = (token, 2048-column slice), one warp each.  With top_k <= 32
// lanes 0..top_k-1 fetch the token's sorted rows and weights once per item
// and share them by shuffles; each lane then loads its 16 bytes of each of
// the top_k rows for two 256-column chunks at a time (2 * top_k loads in
// flight) before accumulating in FP32, j ascending.  Larger top_k take the
// same steps in batches of 32 ids.
constexpr int kCBatch = 8;
constexpr int kCCols = 2048;

__device__ __forceinline__ void combine_acc(float (&acc)[8], const uint4 v, float w) {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, __uint_as_float(w4[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, __uint_as_float(w4[i] & 0xFFFF0000u), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ uint4 combine_pack(const float (&acc)[8]) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[i] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]))) |
               (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1])))
                << 16);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void combine_topk_kernel(const uint16_t* __restrict__ y,
                                    const int32_t* __restrict__ src_to_sorted,
                                    const float* __restrict__ weights, int M, int top_k, int N,
                                    uint16_t* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int ncs = (N + kCCols - 1) / kCCols;
    const long long items = static_cast<long long>(M) * ncs;
    for (long long item = gw; item < items; item += nw) {
        const int t = static_cast<int>(item / ncs);
        const int cbeg = static_cast<int>(item % ncs) * kCCols;
        const int cend = min(N, cbeg + kCCols);
        const int32_t* rows_t = src_to_sorted + static_cast<long long>(t) * top_k;
        const float* w_t = weights + static_cast<long long>(t) * top_k;
        // the first 32 ids once per item (all of them when top_k <= 32)
        int first_r = -1;
        float first_w = 0.0f;
        if (lane < top_k) {
            first_r = __ldg(rows_t + lane);
            first_w = __ldg(w_t + lane);
        }
        for (int n0 = cbeg + 8 * lane; n0 < cend; n0 += 512) {
            const int n1 = n0 + 256;
            const bool two = n1 < cend;
            float acc0[8], acc1[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc0[i] = acc1[i] = 0.0f;
            for (int j0 = 0; j0 < top_k; j0 += 32) {
                int my_r = first_r;
                float my_w = first_w;
                if (j0 > 0) {
                    my_r = -1;
                    my_w = 0.0f;
                    if (j0 + lane < top_k) {
                        my_r = __ldg(rows_t + j0 + lane);
                        my_w = __ldg(w_t + j0 + lane);
                    }
                }
                const int nj = min(32, top_k - j0);
                for (int b0 = 0; b0 < nj; b0 += kCBatch) {
                    uint4 v0[kCBatch], v1[kCBatch];
                    float wj[kCBatch];
#pragma unroll
                    for (int jj = 0; jj < kCBatch; ++jj) {
                        const int r = __shfl_sync(0xFFFFFFFFu, my_r, (b0 + jj) & 31);
                        wj[jj] = __shfl_sync(0xFFFFFFFFu, my_w, (b0 + jj) & 31);
                        v0[jj] = v1[jj] = make_uint4(0, 0, 0, 0);
                        if (b0 + jj < nj && r >= 0) {
                            const uint16_t* yr = y + static_cast<long long>(r) * N;
                            v0[jj] = __ldg(reinterpret_cast<const uint4*>(yr + n0));
                            if (two) v1[jj] = __ldg(reinterpret_cast<const uint4*>(yr + n1));
                        } else {
                            wj[jj] = 0.0f;
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < kCBatch; ++jj) {
                        if (b0 + jj >= nj) break;
                        combine_acc(acc0, v0[jj], wj[jj]);
                        combine_acc(acc1, v1[jj], wj[jj]);
                    }
                }
            }
            uint16_t* ot = out + static_cast<long long>(t) * N;
            *reinterpret_cast<uint4*>(ot + n0) = combine_pack(acc0);
            if (two) *reinterpret_cast<uint4*>(ot + n1) = combine_pack(acc1);
        }
    }
}

}  // namespace

cudaError_t launch_quantize_gather(const uint16_t* x, int K, int top_k, const int32_t* s2d,
                                   int rows, uint8_t* a_fp8, uint8_t* a_scale, int num_sms,
                                   cudaStream_t stream) {
    long long blocks = rows;                         // one sorted row per block and pass
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    quantize_gather_kernel<<<static_cast<int>(blocks), kQThreads, 0, stream>>>(
        x, K, top_k, s2d, rows, a_fp8, a_scale);
    return cudaGetLastError();
}

cudaError_t launch_quantize_scatter(const uint16_t* x, int M, int K, int top_k, const int32_t* d2s,
                                    int rows, uint8_t* a_fp8, uint8_t* a_scale, int num_sms,
                                    cudaStream_t stream) {
    long long blocks = M;                            // one token per block and pass
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    quantize_scatter_kernel<<<static_cast<int>(blocks), kQThreads, 0, stream>>>(
        x, M, K, top_k, d2s, rows, a_fp8, a_scale);
    return cudaGetLastError();
}

int quantize_scatter_max_top_k() { return kMaxScatterTopK; }

cudaError_t launch_combine_topk(const uint16_t* y, const int32_t* d2s, const float* weights,
                                int M, int top_k, int N, uint16_t* out, int num_sms,
                                cudaStream_t stream) {
    const long long items = static_cast<long long>(M) * ((N + kCCols - 1) / kCCols);
    long long blocks = (items + 7) / 8;              // 256 threads = 8 work items per pass
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    combine_topk_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(y, d2s, weights, M, top_k,
                                                                     N, out);
    return cudaGetLastError();
}

}  // namespace hg
