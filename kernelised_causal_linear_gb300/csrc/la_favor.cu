// la_favor.cu -- positive random features (Performer, FAVOR+).
//
// For rows u of length d and r Gaussian rows w_j (drawn by the caller, e.g.
// orthogonal blocks):
//
//   x = u / d^(1/4),   phi(u)_j = exp(w_j . x - |x|^2 / 2) / sqrt(r)
//
// so that phi(q) . phi(k) estimates exp(q . k / sqrt(d)) without bias
// ("Efficient Attention Variants", section 6: the exponential kernel as an
// expectation over Gaussian w; the features are positive, so the normalised
// linear-attention read keeps a positive denominator).  The features then go
// through la_forward with the identity-normalised map (r = the feature
// dimension of the state).
//
// The kernel is one streaming pass (read u, write phi(u)); W^T sits in shared
// memory, one warp takes one row at a time: its lanes hold x (strided), the
// norm is a warp reduction, and lane l computes the features l, l + 32, ...
#include <math.h>

#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxR = 256;
constexpr int kMaxD = 128;

template <typename TI, typename TO>
__global__ void __launch_bounds__(kWarps * 32)
    k_favor(const TI* __restrict__ x, const float* __restrict__ w, TO* __restrict__ out,
            int64_t rows, int d, int r)
{
    extern __shared__ float wt[];  // [d][r]: wt[c * r + j] = w[j * d + c]
    for (int e = threadIdx.x; e < d * r; e += blockDim.x) {
        const int j = e / d, c = e % d;
        wt[c * r + j] = w[e];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float s = 1.0f / sqrtf(sqrtf((float)d));  // d^(-1/4)
    const float inv_sqrt_r = 1.0f / sqrtf((float)r);
    for (int64_t row = (int64_t)blockIdx.x * kWarps + warp; row < rows;
         row += (int64_t)gridDim.x * kWarps) {
        // lane l holds x_c for c = l, l + 32, ... (d <= 128: up to 4)
        float xr[kMaxD / 32];
        float nrm = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxD / 32; ++i) {
            const int c = lane + 32 * i;
            xr[i] = c < d ? to_f32<TI>(x[row * d + c]) * s : 0.f;
            nrm = fmaf(xr[i], xr[i], nrm);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            nrm += __shfl_xor_sync(0xffffffffu, nrm, o);
        float acc[kMaxR / 32];
#pragma unroll
        for (int i = 0; i < kMaxR / 32; ++i)
            acc[i] = 0.f;
#pragma unroll
        for (int ci = 0; ci < kMaxD / 32; ++ci) {
            if (32 * ci >= d)
                break;
            for (int l = 0; l < 32; ++l) {
                const int c = 32 * ci + l;
                const float xc = __shfl_sync(0xffffffffu, xr[ci], l);
                if (c >= d)
                    break;
#pragma unroll
                for (int i = 0; i < kMaxR / 32; ++i) {
                    const int j = lane + 32 * i;
                    if (j < r)
                        acc[i] = fmaf(wt[c * r + j], xc, acc[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kMaxR / 32; ++i) {
            const int j = lane + 32 * i;
            if (j < r) {
                const float f = expf(acc[i] - 0.5f * nrm) * inv_sqrt_r;
                if constexpr (sizeof(TO) == 2)
                    out[row * r + j] = __float2bfloat16_rn(f);
                else
                    out[row * r + j] = f;
            }
        }
    }
}

template <typename TI, typename TO>
cudaError_t launch(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                   cudaStream_t st)
{
    const size_t smem = sizeof(float) * (size_t)d * r;
    cudaError_t e = cudaFuncSetAttribute(k_favor<TI, TO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (rows + kWarps - 1) / kWarps;
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    k_favor<TI, TO><<<grid, kWarps * 32, smem, st>>>(static_cast<const TI*>(x), w,
                                                     static_cast<TO*>(out), rows, d, r);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool favor_shape_ok(int d, int r) { return d >= 1 && d <= kMaxD && r >= 1 && r <= kMaxR; }

cudaError_t favor_features(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                           int in_dtype, int out_dtype, cudaStream_t st)
{
    if (in_dtype == LA_BF16)
        return out_dtype == LA_BF16 ? launch<__nv_bfloat16, __nv_bfloat16>(x, w, out, rows, d, r, st)
                                    : launch<__nv_bfloat16, float>(x, w, out, rows, d, r, st);
    return out_dtype == LA_BF16 ? launch<float, __nv_bfloat16>(x, w, out, rows, d, r, st)
                                : launch<float, float>(x, w, out, rows, d, r, st);
}

}  // namespace la
