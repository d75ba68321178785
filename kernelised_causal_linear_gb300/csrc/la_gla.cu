// la_gla.cu -- causal linear attention with a per-key-channel decay (GLA).
//
//   S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T,   z_t = alpha_t o z_{t-1} + phi(k_t)
//   o_t = phi(q_t)^T S_t / phi(q_t)^T z_t     (o_t = phi(q_t)^T S_t unnormalised)
//
// alpha_t in (0, 1]^d scales row i of the state (key channel i) and is
// broadcast along the value channels ("Efficient Attention Variants", section
// 7.2 GLA; "Linear Attention and SSM", the RWKV-5/6 state M_s = diag(w)
// M_{s-1} + k_s^T v_s).  The gates are inputs (data dependent, drawn or
// computed by the caller).
//
// Chunked on CUDA cores in fp32, in three launches like the scalar-decay
// path, with every decay factor taken as exp of a difference of running
// log-sums, so that no factor exceeds 1 (no ratio of small products):
//   1. block state   dS_b = sum_t exp(L_end - L_t) o phi(k_t) v_t^T, with L the
//                    running sum of log alpha inside the block; the block's
//                    total decay exp(L_end) per channel is stored beside it
//   2. block scan    P_{b+1} = diag(exp(L_end,b)) P_b + dS_b
//   3. block output  sub-chunks of kSub tokens in order with the running state
//                    in shared memory:
//                      inter  (phi(q_t) o exp(L_t - L_{m-1}))^T S
//                      intra  A_tj = sum_i phi(q_t)_i phi(k_j)_i exp(L_t,i - L_j,i), j <= t
//                    then S <- diag(exp(L_end - L_{m-1})) S + sum_j (phi(k_j) o exp(L_end - L_j)) v_j^T
//                    (m = the sub-chunk's first token, L running from the
//                    sub-chunk's start).
#include <float.h>
#include <math.h>

#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kBlockL = 128;  // tokens per block
constexpr int kSub = 32;      // tokens per sub-chunk

template <typename T>
__device__ __forceinline__ float ldf(const T* p)
{
    return to_f32<T>(*p);
}

// ------------------------------------------------------------- step 1 ----
// Thread (ti, tj) owns RI rows (channels) x 4 value columns of the D x DV
// block state.  The running log-sum of each channel is kept by thread i < D.
template <int D, int DV, typename T>
__global__ void __launch_bounds__(kThreads)
    k_gla_state(const T* __restrict__ kp, const T* __restrict__ vp, const float* __restrict__ ap,
                float* __restrict__ ws, float* __restrict__ dec, int64_t N, int nblk, int fm)
{
    constexpr int TJ = (DV / 4) < 32 ? (DV / 4) : 32;
    constexpr int TI = kThreads / TJ;
    constexpr int RI = D / TI;
    __shared__ __align__(16) float sk[kSub][D];  // phi(k) o exp(L_end - L_t)
    __shared__ __align__(16) float sv[kSub][DV];
    __shared__ float slog[D];                    // L_end of the block per channel
    const int64_t gb = blockIdx.x;
    const int64_t seq = gb / nblk;
    const int blk = (int)(gb % nblk);
    const int64_t t0 = (int64_t)blk * kBlockL;
    const int len = (int)min((int64_t)kBlockL, N - t0);
    const T* kb = kp + (seq * N + t0) * D;
    const T* vb = vp + (seq * N + t0) * DV;
    const float* ab = ap + (seq * N + t0) * D;
    const int tid = threadIdx.x, tj = tid % TJ, ti = tid / TJ;

    // total log decay of the block per channel
    if (tid < D) {
        float l = 0.f;
        for (int t = 0; t < len; ++t)
            l += logf(ab[(int64_t)t * D + tid]);
        slog[tid] = l;
    }
    float run = 0.f;  // L_t of channel tid (tid < D), running
    __syncthreads();
    float acc[RI][4];
#pragma unroll
    for (int a = 0; a < RI; ++a)
        acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
    float zacc = 0.f;
    for (int s0 = 0; s0 < len; s0 += kSub) {
        const int n = min(kSub, len - s0);
        if (tid < D) {
            for (int t = 0; t < kSub; ++t) {
                float x = 0.f;
                if (t < n) {
                    run += logf(ab[(int64_t)(s0 + t) * D + tid]);
                    x = phi_f32(ldf(kb + (int64_t)(s0 + t) * D + tid), fm) * expf(slog[tid] - run);
                }
                sk[t][tid] = x;
            }
        }
        for (int e = tid; e < kSub * DV; e += kThreads) {
            const int t = e / DV, c = e % DV;
            sv[t][c] = t < n ? ldf(vb + (int64_t)(s0 + t) * DV + c) : 0.f;
        }
        __syncthreads();
        for (int t = 0; t < kSub; ++t) {
            const float4 vv = *reinterpret_cast<const float4*>(&sv[t][tj * 4]);
#pragma unroll
            for (int a = 0; a < RI; ++a) {
                const float f = sk[t][ti + a * TI];
                acc[a][0] = fmaf(f, vv.x, acc[a][0]);
                acc[a][1] = fmaf(f, vv.y, acc[a][1]);
                acc[a][2] = fmaf(f, vv.z, acc[a][2]);
                acc[a][3] = fmaf(f, vv.w, acc[a][3]);
            }
            if (tid < D)
                zacc += sk[t][tid];
        }
        __syncthreads();
    }
    float* dst = ws + gb * (int64_t)(D * DV + D);
#pragma unroll
    for (int a = 0; a < RI; ++a) {
        const int i = ti + a * TI;
        *reinterpret_cast<float4*>(dst + i * DV + tj * 4) =
            make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    }
    if (tid < D) {
        dst[D * DV + tid] = zacc;
        dec[gb * D + tid] = expf(slog[tid]);
    }
}

// ------------------------------------------------------------- step 2 ----
// Exclusive prefix over the blocks of each sequence, in place: element e of
// the state (row i = e / DV, or the normaliser entry i) decays by the block's
// exp(L_end) of channel i.
__global__ void __launch_bounds__(kThreads)
    k_gla_scan(float* __restrict__ ws, const float* __restrict__ dec, int nblk, int D, int DV)
{
    const int E = D * DV + D;
    const int per_seq = (E + kThreads - 1) / kThreads;
    const int64_t seq = blockIdx.x / per_seq;
    const int e = (int)(blockIdx.x % per_seq) * kThreads + threadIdx.x;
    if (e >= E)
        return;
    const int row = e < D * DV ? e / DV : e - D * DV;
    float* base = ws + seq * (int64_t)nblk * E + e;
    const float* db = dec + seq * (int64_t)nblk * D + row;
    float acc = 0.f;
    for (int b = 0; b < nblk; ++b) {
        const float x = base[(int64_t)b * E];
        base[(int64_t)b * E] = acc;
        acc = fmaf(acc, db[(int64_t)b * D], x);
    }
}

// ------------------------------------------------------------- step 3 ----
template <int D, int DV>
struct GlaSmem {
    static constexpr size_t floats = (size_t)D * DV + D      // S, z
                                     + 3 * (size_t)kSub * D  // phi(q), phi(k), L (running log)
                                     + (size_t)kSub * DV     // v
                                     + (size_t)kSub * (kSub + 1) + kSub;  // A, den
    static constexpr size_t bytes = floats * sizeof(float);
};

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kThreads)
    k_gla_out(const T* __restrict__ qp, const T* __restrict__ kp, const T* __restrict__ vp,
              const float* __restrict__ ap, float* __restrict__ out, const float* __restrict__ ws,
              int64_t N, int nblk, int fm)
{
    extern __shared__ __align__(16) float smem[];
    float* sS = smem;
    float* sz = sS + D * DV;
    float* sq = sz + D;
    float* sk = sq + kSub * D;
    float* sL = sk + kSub * D;
    float* sv = sL + kSub * D;
    float* sA = sv + kSub * DV;
    float* sden = sA + kSub * (kSub + 1);
    constexpr int LDA = kSub + 1;
    constexpr int E = D * DV + D;
    constexpr int TJo = (DV / 4) < 32 ? (DV / 4) : 32;
    constexpr int TIo = kThreads / TJo;
    constexpr int RIo = (kSub + TIo - 1) / TIo;
    constexpr int TJ = TJo, TI = TIo, RI = D / TI;

    const int64_t gb = blockIdx.x;
    const int64_t seq = gb / nblk;
    const int blk = (int)(gb % nblk);
    const int64_t t0 = (int64_t)blk * kBlockL;
    const int len = (int)min((int64_t)kBlockL, N - t0);
    const int tid = threadIdx.x;
    const bool norm = fm_normalised(fm);
    for (int e = tid; e < E; e += kThreads)
        sS[e] = ws[gb * E + e];  // sz follows sS
    const T* qb = qp + (seq * N + t0) * D;
    const T* kb = kp + (seq * N + t0) * D;
    const T* vb = vp + (seq * N + t0) * DV;
    const float* ab = ap + (seq * N + t0) * D;
    float* ob = out + (seq * N + t0) * DV;

    for (int s0 = 0; s0 < len; s0 += kSub) {
        const int n = min(kSub, len - s0);
        __syncthreads();  // the previous sub-chunk is consumed
        if (tid < D) {    // running log decay of channel tid from the sub-chunk's start
            float run = 0.f;
            for (int t = 0; t < kSub; ++t) {
                if (t < n)
                    run += logf(ab[(int64_t)(s0 + t) * D + tid]);
                sL[t * D + tid] = run;
            }
        }
        for (int e = tid; e < kSub * D; e += kThreads) {
            const int t = e / D, i = e % D;
            const bool in = t < n;
            sq[e] = in ? phi_f32(ldf(qb + (int64_t)(s0 + t) * D + i), fm) : 0.f;
            sk[e] = in ? phi_f32(ldf(kb + (int64_t)(s0 + t) * D + i), fm) : 0.f;
        }
        for (int e = tid; e < kSub * DV; e += kThreads) {
            const int t = e / DV, c = e % DV;
            sv[e] = t < n ? ldf(vb + (int64_t)(s0 + t) * DV + c) : 0.f;
        }
        // When the sub-chunk's decay stays above e^-60 in every channel (thread
        // tid < D tests its own channel, written above by itself),
        // exp(L_t - L_j) = exp(L_t) exp(-L_j) with both factors in fp32 range:
        // phi(q) and phi(k) are rescaled once and the scores are plain dot
        // products; otherwise every factor is taken as exp of a difference.
        const bool split =
            __syncthreads_and(tid >= D || sL[(n - 1) * D + tid] >= -60.0f) != 0;
        if (split) {
            for (int e = tid; e < kSub * D; e += kThreads) {
                sq[e] *= expf(sL[e]);
                sk[e] *= expf(-sL[e]);
            }
            __syncthreads();
        }
        // intra scores with the per-channel decay between the two tokens
        for (int e = tid; e < kSub * kSub; e += kThreads) {
            const int t = e / kSub, j = e % kSub;
            float a = 0.f;
            if (j <= t) {
                const float* x = sq + t * D;
                const float* y = sk + j * D;
                const float* lt = sL + t * D;
                const float* lj = sL + j * D;
                if (split)
                    for (int i = 0; i < D; ++i)
                        a = fmaf(x[i], y[i], a);
                else
                    for (int i = 0; i < D; ++i)
                        a = fmaf(x[i] * y[i], __expf(lt[i] - lj[i]), a);
            }
            sA[t * LDA + j] = a;
        }
        __syncthreads();
        // denominators: (phi(q_t) o exp(L_t)) . z + sum_j A_tj
        if (tid < kSub) {
            const int t = tid;
            float den = 0.f;
            for (int i = 0; i < D; ++i)
                den = fmaf(split ? sq[t * D + i] : sq[t * D + i] * __expf(sL[t * D + i]), sz[i],
                           den);
            for (int j = 0; j <= t; ++j)
                den += sA[t * LDA + j];
            sden[t] = den;
        }
        __syncthreads();
        {
            const int tj = tid % TJo, ti = tid / TJo;
            for (int a = 0; a < RIo; ++a) {
                const int t = ti + a * TIo;
                if (t >= kSub)
                    break;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int i = 0; i < D; ++i) {
                    const float f = split ? sq[t * D + i] : sq[t * D + i] * __expf(sL[t * D + i]);
                    const float4 s = *reinterpret_cast<const float4*>(sS + i * DV + tj * 4);
                    acc.x = fmaf(f, s.x, acc.x);
                    acc.y = fmaf(f, s.y, acc.y);
                    acc.z = fmaf(f, s.z, acc.z);
                    acc.w = fmaf(f, s.w, acc.w);
                }
                for (int j = 0; j <= t; ++j) {
                    const float wgt = sA[t * LDA + j];
                    const float4 vv = *reinterpret_cast<const float4*>(sv + j * DV + tj * 4);
                    acc.x = fmaf(wgt, vv.x, acc.x);
                    acc.y = fmaf(wgt, vv.y, acc.y);
                    acc.z = fmaf(wgt, vv.z, acc.z);
                    acc.w = fmaf(wgt, vv.w, acc.w);
                }
                if (t < n) {
                    if (norm) {
                        const float inv = 1.0f / fmaxf(sden[t], FLT_MIN);
                        acc.x *= inv, acc.y *= inv, acc.z *= inv, acc.w *= inv;
                    }
                    *reinterpret_cast<float4*>(ob + (int64_t)(s0 + t) * DV + tj * 4) = acc;
                }
            }
        }
        __syncthreads();  // every read of S, z for this sub-chunk is done
        // S <- diag(exp(L_end)) S + sum_j (phi(k_j) o exp(L_end - L_j)) v_j^T ; z alike
        {
            const int tj = tid % TJ, ti = tid / TJ;
            for (int a = 0; a < RI; ++a) {
                const int i = ti + a * TI;
                const float lend = sL[(n - 1) * D + i];
                const float gi = expf(lend);
                float4 s = *reinterpret_cast<float4*>(sS + i * DV + tj * 4);
                s.x *= gi, s.y *= gi, s.z *= gi, s.w *= gi;
                for (int j = 0; j < n; ++j) {
                    const float f = split ? sk[j * D + i] * gi
                                          : sk[j * D + i] * __expf(lend - sL[j * D + i]);
                    const float4 vv = *reinterpret_cast<const float4*>(sv + j * DV + tj * 4);
                    s.x = fmaf(f, vv.x, s.x);
                    s.y = fmaf(f, vv.y, s.y);
                    s.z = fmaf(f, vv.z, s.z);
                    s.w = fmaf(f, vv.w, s.w);
                }
                *reinterpret_cast<float4*>(sS + i * DV + tj * 4) = s;
            }
            if (tid < D) {
                const float lend = sL[(n - 1) * D + tid];
                const float gz = expf(lend);
                float zz = sz[tid] * gz;
                for (int j = 0; j < n; ++j)
                    zz = fmaf(sk[j * D + tid], split ? gz : __expf(lend - sL[j * D + tid]), zz);
                sz[tid] = zz;
            }
        }
    }
}

int gla_blocks(int64_t N) { return (int)((N + kBlockL - 1) / kBlockL); }

template <int D, int DV, typename T>
cudaError_t run_gla(const GlaArgs& a)
{
    const int64_t BH = a.B * a.H;
    const int nblk = gla_blocks(a.N);
    const int E = D * DV + D;
    float* ws = static_cast<float*>(a.ws);
    float* dec = ws + BH * (int64_t)nblk * E;  // [BH][nblk][D]
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    k_gla_state<D, DV, T><<<(unsigned)(BH * nblk), kThreads, 0, a.stream>>>(k, v, a.alpha, ws, dec,
                                                                           a.N, nblk, a.fm);
    count_launches(1);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    const int per_seq = (E + kThreads - 1) / kThreads;
    k_gla_scan<<<(unsigned)(BH * per_seq), kThreads, 0, a.stream>>>(ws, dec, nblk, D, DV);
    count_launches(1);
    err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    const size_t smem = GlaSmem<D, DV>::bytes;
    auto kern = k_gla_out<D, DV, T>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    kern<<<(unsigned)(BH * nblk), kThreads, smem, a.stream>>>(q, k, v, a.alpha, a.out, ws, a.N,
                                                              nblk, a.fm);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

size_t gla_workspace(int64_t BH, int64_t N, int d, int dv)
{
    if (N <= 0)
        return 0;
    const size_t nblk = (size_t)gla_blocks(N);
    return sizeof(float) * (size_t)BH * nblk * ((size_t)d * dv + d + d);
}

cudaError_t gla_forward(const GlaArgs& a)
{
    const bool bf = a.dtype == LA_BF16;
#define LA_GLA_CASE(D_, DV_) \
    case D_ * 1000 + DV_: return bf ? run_gla<D_, DV_, __nv_bfloat16>(a) : run_gla<D_, DV_, float>(a);
    switch (a.d * 1000 + a.dv) {
        LA_GLA_CASE(32, 32)
        LA_GLA_CASE(32, 64)
        LA_GLA_CASE(32, 128)
        LA_GLA_CASE(64, 32)
        LA_GLA_CASE(64, 64)
        LA_GLA_CASE(64, 128)
        LA_GLA_CASE(128, 32)
        LA_GLA_CASE(128, 64)
        LA_GLA_CASE(128, 128)
    default:
        return cudaErrorInvalidValue;
    }
#undef LA_GLA_CASE
}

}  // namespace la
