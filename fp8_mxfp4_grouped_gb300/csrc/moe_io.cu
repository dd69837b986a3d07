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

// One half-warp per 128-element group: lane j of the half holds elements
// 8j .. 8j+7 (one 16-byte load, one 8-byte store).
__global__ void quantize_gather_kernel(const uint16_t* __restrict__ x, int K, int top_k,
                                       const int32_t* __restrict__ sorted_to_src, int rows,
                                       uint8_t* __restrict__ a_fp8, uint8_t* __restrict__ a_scale) {
    const int groups_per_row = K / kGroup;
    const long long total = static_cast<long long>(rows) * groups_per_row;
    const int half = (threadIdx.x >> 4) & 1;
    const int j = threadIdx.x & 15;
    const long long stride = static_cast<long long>(gridDim.x) * (blockDim.x >> 4);
    for (long long gi = static_cast<long long>(blockIdx.x) * (blockDim.x >> 4) + (threadIdx.x >> 4);
         gi - half < total; gi += stride) {
        // both halves of a warp iterate together; a half past the end idles
        const bool active = gi < total;
        long long r = 0;
        int g = 0, src = -1;
        if (active) {
            r = gi / groups_per_row;
            g = static_cast<int>(gi - r * groups_per_row);
            src = __ldg(sorted_to_src + r);
        }
        const bool live = active && src >= 0;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (live) {
            const long long t = src / top_k;
            v = __ldg(reinterpret_cast<const uint4*>(x + t * K + g * kGroup) + j);
        }
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
        if (!live) continue;
        uint8_t code_scale;
        uint32_t lo = 0, hi = 0;
        if (nonfinite) {
            code_scale = 0xFF;                       // E8M0 NaN
            lo = hi = 0x7F7F7F7Fu;                   // E4M3 NaN
        } else {
            const int e = scale_exponent(amax);
            code_scale = static_cast<uint8_t>(127 + e);
            // 2^-e from its bits: finite BF16 inputs give e <= 120, so the
            // biased exponent 127 - e stays in [7, 254] (a normal float).
            const float inv = __int_as_float((127 - e) << 23);
            uint32_t b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                b[i] = __nv_cvt_float_to_fp8(f[i] * inv, __NV_SATFINITE, __NV_E4M3);
            }
            lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
            hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
        }
        uint8_t* dst = a_fp8 + r * K + g * kGroup + 8 * j;
        *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
        if (j == 0) a_scale[r * groups_per_row + g] = code_scale;
    }
}

// One warp per token, 8 output columns (16 bytes) per lane per step.
__global__ void combine_topk_kernel(const uint16_t* __restrict__ y,
                                    const int32_t* __restrict__ src_to_sorted,
                                    const float* __restrict__ weights, int M, int top_k, int N,
                                    uint16_t* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < M; t += gridDim.x * warps) {
        for (int n0 = 8 * lane; n0 < N; n0 += 256) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            for (int jj = 0; jj < top_k; ++jj) {
                const int r = __ldg(src_to_sorted + static_cast<long long>(t) * top_k + jj);
                if (r < 0) continue;
                const float wgt = __ldg(weights + static_cast<long long>(t) * top_k + jj);
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(y + static_cast<long long>(r) * N + n0));
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = fmaf(wgt, __uint_as_float(w4[i] << 16), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(wgt, __uint_as_float(w4[i] & 0xFFFF0000u), acc[2 * i + 1]);
                }
            }
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[i] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]))) |
                       (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1])))
                        << 16);
            }
            *reinterpret_cast<uint4*>(out + static_cast<long long>(t) * N + n0) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

}  // namespace

cudaError_t launch_quantize_gather(const uint16_t* x, int K, int top_k, const int32_t* s2d,
                                   int rows, uint8_t* a_fp8, uint8_t* a_scale, int num_sms,
                                   cudaStream_t stream) {
    const long long groups = static_cast<long long>(rows) * (K / kGroup);
    long long blocks = (groups + 15) / 16;           // 256 threads = 16 groups per pass
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    quantize_gather_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(x, K, top_k, s2d, rows,
                                                                       a_fp8, a_scale);
    return cudaGetLastError();
}

cudaError_t launch_combine_topk(const uint16_t* y, const int32_t* d2s, const float* weights,
                                int M, int top_k, int N, uint16_t* out, int num_sms,
                                cudaStream_t stream) {
    long long blocks = (M + 7) / 8;                   // 256 threads = 8 tokens per pass
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) return cudaSuccess;
    combine_topk_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(y, d2s, weights, M, top_k,
                                                                     N, out);
    return cudaGetLastError();
}

}  // namespace hg
