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
// The exponent is a small fp32 matrix product X W^T (K = d <= 128), kept in
// fp32 on the CUDA cores: a bf16 W would move the exponent by |x||w| 2^-9,
// about 1 % of the feature.  A persistent CTA holds W^T in shared memory and
// takes tiles of kTileRows rows; each thread owns 8 rows x 4 consecutive
// features of a 128-feature block (three 16-byte shared loads per 32 FMAs),
// and the row norms come from the same staged tile.
#include <math.h>

#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kTileRows = 64;
constexpr int kBlockCols = 128;        // features per pass of the thread block
constexpr int kLdx = kTileRows + 4;    // row stride of the staged X^T tile
constexpr int kMaxR = 256;
constexpr int kMaxD = 128;

__host__ __device__ constexpr int ld_w(int r)
{
    return (r + kBlockCols - 1) / kBlockCols * kBlockCols + 4;
}

// W^T, the staged tile (fp32, transposed), and the raw next tile
__host__ __device__ constexpr size_t smem_bytes(int d, int r, int esz)
{
    return sizeof(float) * ((size_t)d * ld_w(r) + (size_t)d * kLdx) + (size_t)kTileRows * d * esz;
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Four consecutive features of one row (16-byte aligned for fp32, 8-byte
// for bf16).
template <typename TO>
__device__ __forceinline__ void store4(TO* dst, const float (&v)[4])
{
    if constexpr (sizeof(TO) == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(dst) = u;
    }
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads)
    k_favor(const TI* __restrict__ x, const float* __restrict__ w, TO* __restrict__ out,
            int64_t rows, int d, int r)
{
    extern __shared__ float4 smem4[];
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const int ldw = ld_w(r);
    float* wt = reinterpret_cast<float*>(smem4);  // [d][ldw]: wt[c * ldw + j] = w[j * d + c]
    float* xt = wt + (size_t)d * ldw;             // [d][kLdx]: the tile's x, transposed
    TI* raw = reinterpret_cast<TI*>(xt + (size_t)d * kLdx);  // [kTileRows][d]: the next tile
    // rows of 16-byte vectors: copied asynchronously while the previous tile
    // is computed (else staged with plain loads)
    constexpr int VW = 16 / (int)sizeof(TI);
    const bool async = d % VW == 0;
    const int nvec = kTileRows * d / VW;
    auto fetch = [&](int64_t tile) {
        if (!async || tile >= (rows + kTileRows - 1) / kTileRows)
            return;
        const int64_t row0 = tile * kTileRows;
        for (int v = tid; v < nvec; v += kThreads) {
            const int rr = v / (d / VW), cv = v - rr * (d / VW);
            const int64_t row = row0 + rr;
            const TI* src = row < rows ? x + row * d + cv * VW : x;
            cp_async16(raw + (size_t)rr * d + cv * VW, src, row < rows ? 16 : 0);
        }
        cp_async_commit();
    };
    for (int e = tid; e < d * (ldw - 4); e += kThreads) {
        const int j = e / d, c = e - j * d;
        wt[c * ldw + j] = j < r ? w[(size_t)j * d + c] : 0.f;
    }
    const float s = 1.0f / sqrtf(sqrtf((float)d));  // d^(-1/4)
    const float inv_sqrt_r = 1.0f / sqrtf((float)r);
    const bool vec = (r & 3) == 0;
    const int64_t ntiles = (rows + kTileRows - 1) / kTileRows;
    fetch(blockIdx.x);
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t row0 = tile * kTileRows;
        cp_async_wait_all();
        __syncthreads();  // W^T and the raw tile are in; the previous tile's reads are done
        if (async) {
            for (int e = tid; e < kTileRows * d; e += kThreads) {
                const int rr = e / d, c = e - rr * d;
                xt[c * kLdx + rr] = to_f32<TI>(raw[e]) * s;
            }
        } else {
            for (int e = tid; e < kTileRows * d; e += kThreads) {
                const int rr = e / d, c = e - rr * d;
                const int64_t row = row0 + rr;
                xt[c * kLdx + rr] = row < rows ? to_f32<TI>(x[row * d + c]) * s : 0.f;
            }
        }
        __syncthreads();
        fetch(tile + gridDim.x);  // the raw buffer is free again
        // |x|^2 of the warp's 8 rows: lane l sums features l, l + 32, ...,
        // then a butterfly leaves every total in every lane
        float nrm[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            nrm[i] = 0.f;
        for (int c = tx; c < d; c += 32) {
            const float4 xa = *reinterpret_cast<const float4*>(xt + c * kLdx + 8 * ty);
            const float4 xb = *reinterpret_cast<const float4*>(xt + c * kLdx + 8 * ty + 4);
            nrm[0] = fmaf(xa.x, xa.x, nrm[0]), nrm[1] = fmaf(xa.y, xa.y, nrm[1]);
            nrm[2] = fmaf(xa.z, xa.z, nrm[2]), nrm[3] = fmaf(xa.w, xa.w, nrm[3]);
            nrm[4] = fmaf(xb.x, xb.x, nrm[4]), nrm[5] = fmaf(xb.y, xb.y, nrm[5]);
            nrm[6] = fmaf(xb.z, xb.z, nrm[6]), nrm[7] = fmaf(xb.w, xb.w, nrm[7]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                nrm[i] += __shfl_xor_sync(0xffffffffu, nrm[i], o);
        for (int rb = 0; rb < ldw - 4; rb += kBlockCols) {
            float acc[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[i][q] = 0.f;
            const float* wp = wt + rb + 4 * tx;
            const float* xp = xt + 8 * ty;
#pragma unroll 4
            for (int c = 0; c < d; ++c) {
                const float4 w4 = *reinterpret_cast<const float4*>(wp + c * ldw);
                const float4 xa = *reinterpret_cast<const float4*>(xp + c * kLdx);
                const float4 xb = *reinterpret_cast<const float4*>(xp + c * kLdx + 4);
                const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[i][0] = fmaf(xv[i], w4.x, acc[i][0]);
                    acc[i][1] = fmaf(xv[i], w4.y, acc[i][1]);
                    acc[i][2] = fmaf(xv[i], w4.z, acc[i][2]);
                    acc[i][3] = fmaf(xv[i], w4.w, acc[i][3]);
                }
            }
            const int j0 = rb + 4 * tx;
            const int nj = min(4, r - j0);
            if (nj <= 0)
                continue;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t row = row0 + 8 * ty + i;
                if (row >= rows)
                    break;
                const float h = 0.5f * nrm[i];
                float f[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    f[q] = expf(acc[i][q] - h) * inv_sqrt_r;
                if (vec && nj == 4) {
                    store4<TO>(out + row * r + j0, f);
                } else {
                    for (int q = 0; q < nj; ++q) {
                        if constexpr (sizeof(TO) == 4)
                            out[row * r + j0 + q] = f[q];
                        else
                            out[row * r + j0 + q] = __float2bfloat16_rn(f[q]);
                    }
                }
            }
        }
    }
}

template <typename TI, typename TO>
cudaError_t launch(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                   cudaStream_t st)
{
    const size_t smem = smem_bytes(d, r, (int)sizeof(TI));
    cudaError_t e = cudaFuncSetAttribute(k_favor<TI, TO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 148, per_sm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_favor<TI, TO>, kThreads, smem);
    const int64_t tiles = (rows + kTileRows - 1) / kTileRows;
    const int64_t cap = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(tiles < cap ? tiles : cap);
    k_favor<TI, TO><<<grid, kThreads, smem, st>>>(static_cast<const TI*>(x), w,
                                                   static_cast<TO*>(out), rows, d, r);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool favor_shape_ok(int d, int r) { return d >= 1 && d <= kMaxD && r >= 1 && r <= kMaxR; }

cudaError_t favor_features(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                           int in_dtype, int out_dtype, cudaStream_t st)
{
    if (rows == 0)
        return cudaSuccess;
    if (in_dtype == LA_BF16)
        return out_dtype == LA_BF16 ? launch<__nv_bfloat16, __nv_bfloat16>(x, w, out, rows, d, r, st)
                                    : launch<__nv_bfloat16, float>(x, w, out, rows, d, r, st);
    return out_dtype == LA_BF16 ? launch<float, __nv_bfloat16>(x, w, out, rows, d, r, st)
                                : launch<float, float>(x, w, out, rows, d, r, st);
}

}  // namespace la
