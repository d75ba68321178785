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
#include "la_sm100.cuh"
#include "la_tc_common.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tcc;

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

// ---------------------------------------------------------------------------
// Tensor-core form (bf16 x, d in {64, 128}, r a multiple of 16): the exponent
// X W'^T with W' = W d^(-1/4) as an exact sum of three bf16 parts (hi, mid, lo:
// about 2^-24 relative, as fp32), so that x (exact in bf16) times W' is
// accumulated in fp32 by three passes of tcgen05 MMAs per 128-row tile.  The
// exponential and the norm run in an epilogue warpgroup that reads the
// accumulator from tensor memory (two buffers: tile i + 1 accumulates while
// tile i is stored).  Roles: warp 0 loads x tiles by TMA (four stages), warp 1
// issues the MMAs, warps 4-11 the epilogue: two warpgroups (one tensor-memory
// lane per row), each taking every other 16-feature block.
constexpr int kTcThreads = 384;
constexpr int kEpiWarps = 8;
constexpr int kTcStages = 4;

struct FavorTcParams {
    CUtensorMap mx;  // x as [1][rows][d] bf16, boxes of 128 rows x 64 columns
    int64_t rows;
    int d, r;
    float* out32;
    __nv_bfloat16* out16;
    const float* w;
    int* status;
};

struct FavorTcBars {
    uint64_t x_full[kTcStages], x_empty[kTcStages], acc_full[2], acc_empty[2], drain;
    uint32_t tmem;
    int abort;
};

__host__ __device__ constexpr uint32_t favor_tc_wbytes(int d, int r) { return 3u * (uint32_t)r * (uint32_t)d * 2u; }
__host__ __device__ constexpr uint32_t favor_tc_smem(int d, int r)
{
    return 1024 + favor_tc_wbytes(d, r) + kTcStages * (uint32_t)d * 128u * 2u + 1024;
}

__device__ __forceinline__ bool tc_bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    if (mbar_test_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort)
            return false;
        if (globaltimer() - t0 > 2000000000ull) {
            *abort = 1;
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ uint64_t kmaj(uint32_t base, int rows, int kk)
{
    return sdesc_sw128(base + (uint32_t)(kk >> 2) * (uint32_t)rows * 128u + (uint32_t)(kk & 3) * 32u,
                       16, 1024);
}

__global__ void __launch_bounds__(kTcThreads, 1) k_favor_tc(const __grid_constant__ FavorTcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int d = p.d, r = p.r, KB = d / 64;
    unsigned char* wpart = sm;                                  // 3 parts x KB blocks x r rows x 128 B
    unsigned char* xst = sm + favor_tc_wbytes(d, r);            // kTcStages x KB x 16 KiB
    FavorTcBars* m = reinterpret_cast<FavorTcBars*>(xst + kTcStages * KB * 16384);
    volatile int* abort = &m->abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = (p.rows + 127) / 128;
    const float s = 1.0f / sqrtf(sqrtf((float)d));
    if (tid == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(&m->x_full[i], 1);
            mbar_init(&m->x_empty[i], 1 + kEpiWarps);  // the MMAs and the epilogue warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&m->acc_full[i], 1);
            mbar_init(&m->acc_empty[i], kEpiWarps);
        }
        mbar_init(&m->drain, 1);
        m->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.mx);
    }
    // W' = W d^(-1/4) as hi + mid + lo, K-major 128-byte swizzled blocks
    for (int e = tid; e < r * d; e += kTcThreads) {
        const int j = e / d, c = e - j * d;
        const float x = p.w[e] * s;
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const float r1 = x - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
        const uint32_t off = (uint32_t)(c >> 6) * (uint32_t)r * 128u + sw128_off(j, (c & 63) >> 3) +
                             (uint32_t)(c & 7) * 2u;
        const uint32_t part = (uint32_t)r * (uint32_t)d * 2u;
        *reinterpret_cast<__nv_bfloat16*>(wpart + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(wpart + part + off) = mid;
        *reinterpret_cast<__nv_bfloat16*>(wpart + 2 * part + off) = lo;
    }
    fence_proxy_async_smem();
    const uint32_t ncols = 2u * (uint32_t)r <= 64 ? 64u : 2u * (uint32_t)r <= 128 ? 128u
                         : 2u * (uint32_t)r <= 256 ? 256u : 512u;
    if (warp == 0) {
        tmem_alloc(&m->tmem, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = m->tmem;

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------- loads
            const uint64_t pol = policy_evict_first();
            int i = 0;
            int last[kTcStages];
            for (int q = 0; q < kTcStages; ++q)
                last[q] = -1;
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int st = i % kTcStages;
                if (i >= kTcStages && !tc_bounded_wait(&m->x_empty[st], ((i / kTcStages) & 1) ^ 1, abort))
                    break;
                mbar_arrive_expect_tx(&m->x_full[st], (uint32_t)KB * 16384u);
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_3d(xst + (st * KB + kb) * 16384, &p.mx, 64 * kb, (int)(t * 128), 0,
                                &m->x_full[st], pol);
                last[st] = (i / kTcStages) & 1;
            }
            if (*abort)
                for (int q = 0; q < kTcStages; ++q)
                    if (last[q] >= 0) {
                        const uint64_t t0 = globaltimer();
                        while (!mbar_try_wait(&m->x_full[q], (uint32_t)last[q]) &&
                               globaltimer() - t0 < 2000000000ull) {
                        }
                    }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // -------------------------------------------- MMAs
            const uint32_t id = idesc_bf16_f32(128, r, false, false);
            const uint32_t wb = smem_addr(wpart), part = (uint32_t)r * (uint32_t)d * 2u;
            int i = 0;
            bool issued = false;
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int st = i % kTcStages, a = i & 1;
                if (!tc_bounded_wait(&m->x_full[st], (i / kTcStages) & 1, abort))
                    break;
                if (i >= 2 && !tc_bounded_wait(&m->acc_empty[a], ((i >> 1) & 1) ^ 1, abort))
                    break;
                tc_fence_after();
                const uint32_t xa = smem_addr(xst + st * KB * 16384);
                const uint32_t dt = tm + (uint32_t)(a * r);
                for (int pp = 0; pp < 3; ++pp)
                    for (int kk = 0; kk < d / 16; ++kk)
                        mma_bf16_ss(dt, kmaj(xa, 128, kk), kmaj(wb + pp * part, r, kk), id,
                                    (pp | kk) != 0);
                mma_commit(&m->x_empty[st]);
                mma_commit(&m->acc_full[a]);
                issued = true;
            }
            if (issued && *abort) {
                mma_commit(&m->drain);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&m->drain, 0) && globaltimer() - t0 < 2000000000ull) {
                }
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------- epilogue
        const int row_in = (warp & 3) * 32 + lane;  // tensor-memory lane = tile row
        const int half = (warp - 4) >> 2;           // 16-feature blocks half, half + 2, ...
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const float l2e = 1.4426950408889634f;
        const float bias = 0.5f * log2f((float)r);  // log2 sqrt(r)
        int i = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int st = i % kTcStages, a = i & 1;
            // |x'|^2 / 2 of this row from the staged tile, then the stage is
            // released for the loads (the MMAs release it too)
            const bool okx = __all_sync(0xffffffffu, tc_bounded_wait(&m->x_full[st], (i / kTcStages) & 1, abort));
            if (!okx)
                break;
            float nrm = 0.f;
            for (int kb = 0; kb < KB; ++kb) {
                const unsigned char* blk = xst + (st * KB + kb) * 16384;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const uint4 u = *reinterpret_cast<const uint4*>(blk + sw128_off(row_in, c8));
                    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float x0 = __uint_as_float(wv[h] << 16);
                        const float x1 = __uint_as_float(wv[h] & 0xffff0000u);
                        nrm = fmaf(x0, x0, fmaf(x1, x1, nrm));
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&m->x_empty[st]);
            // f_j = exp(acc_j - |x'|^2 / 2) / sqrt(r) = 2^(acc_j l2e - (|x'|^2 / 2) l2e - log2 sqrt r)
            const float off = (0.5f * nrm * s * s) * l2e + bias;
            const bool oka = __all_sync(0xffffffffu, tc_bounded_wait(&m->acc_full[a], (i >> 1) & 1, abort));
            if (!oka)
                break;
            tc_fence_after();
            const int64_t row = t * 128 + row_in;
            const bool live = row < p.rows;
            for (int c0 = 16 * half; c0 < r; c0 += 32) {
                uint32_t v[16];
                tmem_ld16(tm + lane_off + (uint32_t)(a * r + c0), v);
                tmem_ld_wait();
                float f[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    f[e] = exp2f(fmaf(__uint_as_float(v[e]), l2e, -off));
                if (live) {
                    if (p.out32) {
                        float4* o = reinterpret_cast<float4*>(p.out32 + row * r + c0);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            o[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
                    } else {
                        uint4* o = reinterpret_cast<uint4*>(p.out16 + row * r + c0);
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            uint32_t pk[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[8 * q + 2 * h], f[8 * q + 2 * h + 1]);
                                pk[h] = *reinterpret_cast<const uint32_t*>(&b2);
                            }
                            o[q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&m->acc_empty[a]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && m->abort)
        set_status(p.status, LA_ERR_TIMEOUT);
    if (warp == 0)
        tmem_dealloc(tm, ncols);
}

bool favor_tc_ok(int d, int r, int in_dtype)
{
    return in_dtype == LA_BF16 && (d == 64 || d == 128) && r % 16 == 0 && r >= 16 &&
           r <= 256 && favor_tc_smem(d, r) <= 232448;
}

cudaError_t launch_tc(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                      bool out_bf16, int* status, cudaStream_t st)
{
    FavorTcParams p;
    memset(&p, 0, sizeof p);
    if (!tma_map_bf16_3d(&p.mx, x, d, rows, 1))
        return cudaErrorInvalidValue;
    p.rows = rows;
    p.d = d;
    p.r = r;
    p.w = w;
    p.status = status;
    if (out_bf16)
        p.out16 = static_cast<__nv_bfloat16*>(out);
    else
        p.out32 = static_cast<float*>(out);
    const uint32_t smem = favor_tc_smem(d, r);
    cudaError_t e = cudaFuncSetAttribute(k_favor_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    const int sms = device_sm_count() > 0 ? device_sm_count() : 148;
    const int64_t tiles = (rows + 127) / 128;
    const int grid = (int)(tiles < sms ? tiles : sms);
    k_favor_tc<<<grid, kTcThreads, smem, st>>>(p);
    count_launches(1);
    return cudaGetLastError();
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
                           int in_dtype, int out_dtype, int* status, cudaStream_t st)
{
    if (rows == 0)
        return cudaSuccess;
    if (favor_tc_ok(d, r, in_dtype) && rows <= INT32_MAX)
        return launch_tc(x, w, out, rows, d, r, out_dtype == LA_BF16, status, st);
    if (in_dtype == LA_BF16)
        return out_dtype == LA_BF16 ? launch<__nv_bfloat16, __nv_bfloat16>(x, w, out, rows, d, r, st)
                                    : launch<__nv_bfloat16, float>(x, w, out, rows, d, r, st);
    return out_dtype == LA_BF16 ? launch<float, __nv_bfloat16>(x, w, out, rows, d, r, st)
                                : launch<float, float>(x, w, out, rows, d, r, st);
}

}  // namespace la
