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
// memory, one warp takes kRows rows at a time: its lanes hold x (strided), the
// norms are warp reductions, and lane l computes the features l, l + 32, ...
#include <math.h>

#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxR = 256;
constexpr int kMaxD = 128;

// One warp computes kRows rows at a time: every W^T value read from shared
// memory feeds kRows FMAs (lane l holds features l, l + 32, ... of each row).
constexpr int kRows = 8;

template <typename TI, typename TO, int RJ>
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
    for (int64_t row0 = ((int64_t)blockIdx.x * kWarps + warp) * kRows; row0 < rows;
         row0 += (int64_t)gridDim.x * kWarps * kRows) {
        // lane l holds x_c of each row for c = l, l + 32, ... (d <= 128)
        float xr[kRows][kMaxD / 32];
        float nrm[kRows];
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            const int64_t row = row0 + rr;
            nrm[rr] = 0.f;
#pragma unroll
            for (int i = 0; i < kMaxD / 32; ++i) {
                const int c = lane + 32 * i;
                xr[rr][i] = (c < d && row < rows) ? to_f32<TI>(x[row * d + c]) * s : 0.f;
                nrm[rr] = fmaf(xr[rr][i], xr[rr][i], nrm[rr]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                nrm[rr] += __shfl_xor_sync(0xffffffffu, nrm[rr], o);
        }
        float acc[kRows][RJ];
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr)
#pragma unroll
            for (int i = 0; i < RJ; ++i)
                acc[rr][i] = 0.f;
#pragma unroll
        for (int ci = 0; ci < kMaxD / 32; ++ci) {
            if (32 * ci >= d)
                break;
#pragma unroll 4
            for (int l = 0; l < 32; ++l) {
                const int c = 32 * ci + l;
                if (c >= d)
                    break;
                float wj[RJ];
#pragma unroll
                for (int i = 0; i < RJ; ++i) {
                    const int j = lane + 32 * i;
                    wj[i] = j < r ? wt[c * r + j] : 0.f;
                }
#pragma unroll
                for (int rr = 0; rr < kRows; ++rr) {
                    const float xc = __shfl_sync(0xffffffffu, xr[rr][ci], l);
#pragma unroll
                    for (int i = 0; i < RJ; ++i)
                        acc[rr][i] = fmaf(wj[i], xc, acc[rr][i]);
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
            const int64_t row = row0 + rr;
            if (row >= rows)
                break;
#pragma unroll
            for (int i = 0; i < RJ; ++i) {
                const int j = lane + 32 * i;
                if (j < r) {
                    const float f = expf(acc[rr][i] - 0.5f * nrm[rr]) * inv_sqrt_r;
                    if constexpr (sizeof(TO) == 2)
                        out[row * r + j] = __float2bfloat16_rn(f);
                    else
                        out[row * r + j] = f;
                }
            }
        }
    }
}

template <typename TI, typename TO, int RJ>
cudaError_t launch_rj(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                      cudaStream_t st)
{
    const size_t smem = sizeof(float) * (size_t)d * r;
    cudaError_t e = cudaFuncSetAttribute(k_favor<TI, TO, RJ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (rows + kWarps * kRows - 1) / (kWarps * kRows);
    const int grid = (int)(want < (int64_t)sms * 4 ? want : (int64_t)sms * 4);
    k_favor<TI, TO, RJ><<<grid, kWarps * 32, smem, st>>>(static_cast<const TI*>(x), w,
                                                         static_cast<TO*>(out), rows, d, r);
    count_launches(1);
    return cudaGetLastError();
}

// r features need RJ = ceil(r / 32) accumulators per lane and row
template <typename TI, typename TO>
cudaError_t launch(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                   cudaStream_t st)
{
    switch ((r + 31) / 32) {
    case 1: return launch_rj<TI, TO, 1>(x, w, out, rows, d, r, st);
    case 2: return launch_rj<TI, TO, 2>(x, w, out, rows, d, r, st);
    case 3: case 4: return launch_rj<TI, TO, 4>(x, w, out, rows, d, r, st);
    default: return launch_rj<TI, TO, kMaxR / 32>(x, w, out, rows, d, r, st);
    }
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
