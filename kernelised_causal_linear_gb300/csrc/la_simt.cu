// la_simt.cu -- chunked forward on CUDA cores, everything in fp32.
//
// This is the general path: any d, dv in {32, 64, 128}, bf16 or fp32 inputs,
// every feature map, optional per-head decay, causal or not.  It is also the
// whole state reduction behind la_state.  Three launches:
//
//   1. chunk state   per block of kBlockL tokens:
//                      dS_b = sum_j w_j phi(k_j) v_j^T,  dz_b = sum_j w_j phi(k_j)
//                      w_j = gamma^(end_b - j)
//                    ("Linear Attention Kernel", section "Rewrite:
//                     associativity": phi(K)^T V is the only intermediate)
//   2. block scan    exclusive prefix over blocks, P_{b+1} = gamma^len P_b + dS_b
//                    ("Efficient Attention Variants", section 8: blocks pass
//                     history through a state / scan)
//   3. block output  sub-chunks of kSub tokens in order, with the running
//                    state S kept in shared memory:
//                      o_i = [gamma^(i+1) phi(q_i)^T S + sum_{j<=i} gamma^(i-j) (phi(q_i).phi(k_j)) v_j]
//                            / [same with v_j -> 1 and S -> z]
//                    then S <- gamma^n S + sum_j gamma^(n-1-j) phi(k_j) v_j^T
//                    ("Linear Attention and SSM", eq. attn-linssm-ssd: the
//                     intra-chunk part is the masked form ((Q K^T) o L) V)
//
// The non-causal form runs step 1, a total reduction (step 2 in total mode)
// and step 3 without the intra-chunk term and without state updates.
#include <float.h>

#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kBlockL = 128;  // tokens per block = per workspace state
constexpr int kSub = 32;      // tokens per sub-chunk inside a block

// 256 threads laid over a D x DV fp32 tile: TJ threads along the value
// channels (4 contiguous floats each), TI along key features (strided rows).
template <int D, int DV>
struct StateTile {
    static constexpr int TJ = (DV / 4) < 32 ? (DV / 4) : 32;
    static constexpr int TI = kThreads / TJ;
    static constexpr int RI = D / TI;
    static_assert(D % TI == 0, "tile");
};

template <typename T>
__device__ __forceinline__ float ldf(const T* p)
{
    return to_f32<T>(*p);
}

// ---------------------------------------------------------------- step 1 ---
template <int D, int DV, typename T>
__global__ void __launch_bounds__(kThreads)
    k_chunk_state(const T* __restrict__ kp, const T* __restrict__ vp, float* __restrict__ ws,
                  int64_t N, int nblk, int H, int fm, GammaTable g)
{
    using TL = StateTile<D, DV>;
    __shared__ __align__(16) float sk[kSub][D];
    __shared__ __align__(16) float sv[kSub][DV];
    const int64_t gb = blockIdx.x;  // seq * nblk + blk
    const int64_t seq = gb / nblk;
    const int blk = (int)(gb % nblk);
    const int head = (int)(seq % H);
    const int64_t t0 = (int64_t)blk * kBlockL;
    const int len = (int)min((int64_t)kBlockL, N - t0);
    const T* kb = kp + (seq * N + t0) * D;
    const T* vb = vp + (seq * N + t0) * DV;
    const int tid = threadIdx.x, tj = tid % TL::TJ, ti = tid / TL::TJ;

    float acc[TL::RI][4];
#pragma unroll
    for (int a = 0; a < TL::RI; ++a)
        acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
    float zacc = 0.f;

    for (int s0 = 0; s0 < len; s0 += kSub) {
        const int n = min(kSub, len - s0);
        for (int e = tid; e < kSub * D; e += kThreads) {
            const int t = e / D, i = e % D;
            float x = 0.f;
            if (t < n) {
                const float w = gamma_pow(g, head, (float)(len - 1 - (s0 + t)));
                x = phi_f32(ldf(kb + (int64_t)(s0 + t) * D + i), fm) * w;
            }
            sk[t][i] = x;
        }
        for (int e = tid; e < kSub * DV; e += kThreads) {
            const int t = e / DV, c = e % DV;
            sv[t][c] = t < n ? ldf(vb + (int64_t)(s0 + t) * DV + c) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int t = 0; t < kSub; ++t) {
            const float4 vv = *reinterpret_cast<const float4*>(&sv[t][tj * 4]);
#pragma unroll
            for (int a = 0; a < TL::RI; ++a) {
                const float f = sk[t][ti + a * TL::TI];
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
    for (int a = 0; a < TL::RI; ++a) {
        const int i = ti + a * TL::TI;
        *reinterpret_cast<float4*>(dst + i * DV + tj * 4) =
            make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    }
    if (tid < D)
        dst[D * DV + tid] = zacc;
}

// ---------------------------------------------------------------- step 2 ---
// mode 0: exclusive prefix over the blocks of each sequence, in place.
// mode 1: no prefix is written.
// The prefix starts from init_S [BH][D*DV] / init_z [BH][D] (the state before
// the first token) or from zero; the total, if tot_S is given, is written to
// tot_S [BH][D*DV] and tot_z [BH][D] (tot_z == NULL: packed into tot_S as
// [BH][D*DV + D]).
__global__ void __launch_bounds__(kThreads)
    k_block_scan(float* __restrict__ ws, int nblk, int64_t N, int H, int D, int DV, int mode,
                 GammaTable g, const float* init_S, const float* init_z, float* tot_S,
                 float* tot_z)
{
    const int E = D * DV + D;
    const int per_seq = (E + kThreads - 1) / kThreads;
    const int64_t seq = blockIdx.x / per_seq;
    const int e = (int)(blockIdx.x % per_seq) * kThreads + threadIdx.x;
    if (e >= E)
        return;
    const int head = (int)(seq % H);
    float* base = ws + seq * (int64_t)nblk * E + e;
    float acc = 0.f;
    if (init_S)
        acc = e < D * DV ? init_S[seq * (int64_t)(D * DV) + e] : init_z[seq * (int64_t)D + (e - D * DV)];
    constexpr int kBatch = 16;  // independent loads in flight per thread
    for (int b0 = 0; b0 < nblk; b0 += kBatch) {
        float x[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            x[j] = (b0 + j < nblk) ? base[(int64_t)(b0 + j) * E] : 0.f;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int b = b0 + j;
            if (b < nblk) {
                if (mode == 0)
                    base[(int64_t)b * E] = acc;
                const int len = (int)min((int64_t)kBlockL, N - (int64_t)b * kBlockL);
                acc = fmaf(acc, gamma_pow(g, head, (float)len), x[j]);
            }
        }
    }
    if (tot_S) {
        if (!tot_z)
            tot_S[seq * (int64_t)E + e] = acc;
        else if (e < D * DV)
            tot_S[seq * (int64_t)(D * DV) + e] = acc;
        else
            tot_z[seq * (int64_t)D + (e - D * DV)] = acc;
    }
}

// ---------------------------------------------------------------- step 3 ---
template <int D, int DV>
struct OutSmem {
    static constexpr int kS = D * DV;
    static constexpr int kZ = D;
    static constexpr int kQ = kSub * D;
    static constexpr int kK = kSub * D;
    static constexpr int kV = kSub * DV;
    static constexpr int kA = kSub * (kSub + 1);
    static constexpr int kDen = kSub;
    static constexpr size_t bytes = sizeof(float) * (kS + kZ + kQ + kK + kV + kA + kDen);
};

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kThreads)
    k_block_out(const T* __restrict__ qp, const T* __restrict__ kp, const T* __restrict__ vp,
                float* __restrict__ out, const float* __restrict__ ws,
                const float* __restrict__ tot, int64_t N, int nblk, int H, int fm, int causal,
                GammaTable g)
{
    using TL = StateTile<D, DV>;
    using SM = OutSmem<D, DV>;
    extern __shared__ __align__(16) float smem[];
    float* sS = smem;
    float* sz = sS + SM::kS;
    float* sq = sz + SM::kZ;
    float* sk = sq + SM::kQ;
    float* sv = sk + SM::kK;
    float* sA = sv + SM::kV;
    float* sden = sA + SM::kA;
    constexpr int E = D * DV + D;
    constexpr int LDA = kSub + 1;

    const int64_t gb = blockIdx.x;
    const int64_t seq = gb / nblk;
    const int blk = (int)(gb % nblk);
    const int head = (int)(seq % H);
    const int64_t t0 = (int64_t)blk * kBlockL;
    const int len = (int)min((int64_t)kBlockL, N - t0);
    const int tid = threadIdx.x;
    const bool norm = fm_normalised(fm);

    // the state entering this block: exclusive prefix, or the total
    const float* src = causal ? ws + gb * E : tot + seq * E;
    for (int e = tid; e < E; e += kThreads)
        sS[e] = src[e];  // sz follows sS, as in the workspace

    const T* qb = qp + (seq * N + t0) * D;
    const T* kb = kp + (seq * N + t0) * D;
    const T* vb = vp + (seq * N + t0) * DV;
    float* ob = out + (seq * N + t0) * DV;

    // output tile mapping: TJo threads along value channels (float4 each)
    constexpr int TJo = (DV / 4) < 32 ? (DV / 4) : 32;
    constexpr int TIo = kThreads / TJo;
    constexpr int RIo = (kSub + TIo - 1) / TIo;

    for (int s0 = 0; s0 < len; s0 += kSub) {
        const int n = min(kSub, len - s0);
        __syncthreads();  // previous sub-chunk fully consumed
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
        __syncthreads();

        // masked, decayed intra-chunk scores A_ij (causal only)
        if (causal) {
            for (int e = tid; e < kSub * kSub; e += kThreads) {
                const int i = e / kSub, j = e % kSub;
                float a = 0.f;
                if (j <= i) {
                    const float* x = sq + i * D;
                    const float* y = sk + j * D;
#pragma unroll 8
                    for (int r = 0; r < D; ++r)
                        a = fmaf(x[r], y[r], a);
                    a *= gamma_pow(g, head, (float)(i - j));
                }
                sA[i * LDA + j] = a;
            }
        }
        __syncthreads();
        // denominators: gamma^(i+1) phi(q_i).z + sum_j A_ij
        if (tid < kSub) {
            const int i = tid;
            float dz = 0.f;
            for (int r = 0; r < D; ++r)
                dz = fmaf(sq[i * D + r], sz[r], dz);
            float den = causal ? gamma_pow(g, head, (float)(i + 1)) * dz : dz;
            if (causal)
                for (int j = 0; j <= i; ++j)
                    den += sA[i * LDA + j];
            sden[i] = den;
        }
        __syncthreads();
        {
            const int tj = tid % TJo, ti = tid / TJo;
            for (int a = 0; a < RIo; ++a) {
                const int i = ti + a * TIo;
                if (i >= kSub)
                    break;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int r = 0; r < D; ++r) {
                    const float f = sq[i * D + r];
                    const float4 s = *reinterpret_cast<const float4*>(sS + r * DV + tj * 4);
                    acc.x = fmaf(f, s.x, acc.x);
                    acc.y = fmaf(f, s.y, acc.y);
                    acc.z = fmaf(f, s.z, acc.z);
                    acc.w = fmaf(f, s.w, acc.w);
                }
                if (causal) {
                    const float gd = gamma_pow(g, head, (float)(i + 1));
                    acc.x *= gd, acc.y *= gd, acc.z *= gd, acc.w *= gd;
                    for (int j = 0; j <= i; ++j) {
                        const float w = sA[i * LDA + j];
                        const float4 vv = *reinterpret_cast<const float4*>(sv + j * DV + tj * 4);
                        acc.x = fmaf(w, vv.x, acc.x);
                        acc.y = fmaf(w, vv.y, acc.y);
                        acc.z = fmaf(w, vv.z, acc.z);
                        acc.w = fmaf(w, vv.w, acc.w);
                    }
                }
                if (i < n) {
                    if (norm) {
                        const float inv = 1.0f / fmaxf(sden[i], FLT_MIN);
                        acc.x *= inv, acc.y *= inv, acc.z *= inv, acc.w *= inv;
                    }
                    *reinterpret_cast<float4*>(ob + (int64_t)(s0 + i) * DV + tj * 4) = acc;
                }
            }
        }
        if (!causal)
            continue;
        __syncthreads();  // every read of sS / sz for this sub-chunk is done
        // S <- gamma^n S + sum_j gamma^(n-1-j) phi(k_j) v_j^T ; same for z
        {
            const int tj = tid % TL::TJ, ti = tid / TL::TJ;
            const float gn = gamma_pow(g, head, (float)n);
#pragma unroll
            for (int a = 0; a < TL::RI; ++a) {
                const int i = ti + a * TL::TI;
                float4 s = *reinterpret_cast<float4*>(sS + i * DV + tj * 4);
                s.x *= gn, s.y *= gn, s.z *= gn, s.w *= gn;
                for (int j = 0; j < n; ++j) {
                    const float f = sk[j * D + i] * gamma_pow(g, head, (float)(n - 1 - j));
                    const float4 vv = *reinterpret_cast<const float4*>(sv + j * DV + tj * 4);
                    s.x = fmaf(f, vv.x, s.x);
                    s.y = fmaf(f, vv.y, s.y);
                    s.z = fmaf(f, vv.z, s.z);
                    s.w = fmaf(f, vv.w, s.w);
                }
                *reinterpret_cast<float4*>(sS + i * DV + tj * 4) = s;
            }
            if (tid < D) {
                float zz = sz[tid] * gn;
                for (int j = 0; j < n; ++j)
                    zz = fmaf(sk[j * D + tid], gamma_pow(g, head, (float)(n - 1 - j)), zz);
                sz[tid] = zz;
            }
        }
    }
}

int blocks_per_seq(int64_t N) { return (int)((N + kBlockL - 1) / kBlockL); }

template <int D, int DV, typename T>
cudaError_t run_forward(const FwdArgs& a, bool state_only)
{
    const int64_t BH = a.B * a.H;
    const int nblk = blocks_per_seq(a.N);
    const int E = D * DV + D;
    float* ws = static_cast<float*>(a.ws);
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    const int H = (int)a.H;

    k_chunk_state<D, DV, T><<<(unsigned)(BH * nblk), kThreads, 0, a.stream>>>(
        k, v, ws, a.N, nblk, H, a.fm, *a.gamma);
    count_launches(1);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    const int per_seq = (E + kThreads - 1) / kThreads;
    const unsigned scan_grid = (unsigned)(BH * per_seq);
    if (state_only) {
        k_block_scan<<<scan_grid, kThreads, 0, a.stream>>>(ws, nblk, a.N, H, D, DV, 1, *a.gamma,
                                                          a.S0, a.z0, a.S_out, a.z_out);
        count_launches(1);
        return cudaGetLastError();
    }
    float* tot = ws + BH * (int64_t)nblk * E;  // non-causal totals [BH][E]
    if (a.causal)
        k_block_scan<<<scan_grid, kThreads, 0, a.stream>>>(ws, nblk, a.N, H, D, DV, 0, *a.gamma,
                                                          a.S0, a.z0, a.S_out, a.z_out);
    else
        k_block_scan<<<scan_grid, kThreads, 0, a.stream>>>(ws, nblk, a.N, H, D, DV, 1, *a.gamma,
                                                          nullptr, nullptr, tot, nullptr);
    count_launches(1);
    err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    const size_t smem = OutSmem<D, DV>::bytes;
    auto kern = k_block_out<D, DV, T>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    kern<<<(unsigned)(BH * nblk), kThreads, smem, a.stream>>>(q, k, v, a.out, ws, tot, a.N, nblk,
                                                              H, a.fm, a.causal, *a.gamma);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

#define LA_DISPATCH_DIMS(FN, ...)                                                     \
    do {                                                                              \
        const bool bf = a.dtype == LA_BF16;                                           \
        switch (a.d * 1000 + a.dv) {                                                  \
        case 32032: return bf ? FN<32, 32, __nv_bfloat16>(__VA_ARGS__) : FN<32, 32, float>(__VA_ARGS__); \
        case 32064: return bf ? FN<32, 64, __nv_bfloat16>(__VA_ARGS__) : FN<32, 64, float>(__VA_ARGS__); \
        case 32128: return bf ? FN<32, 128, __nv_bfloat16>(__VA_ARGS__) : FN<32, 128, float>(__VA_ARGS__); \
        case 64032: return bf ? FN<64, 32, __nv_bfloat16>(__VA_ARGS__) : FN<64, 32, float>(__VA_ARGS__); \
        case 64064: return bf ? FN<64, 64, __nv_bfloat16>(__VA_ARGS__) : FN<64, 64, float>(__VA_ARGS__); \
        case 64128: return bf ? FN<64, 128, __nv_bfloat16>(__VA_ARGS__) : FN<64, 128, float>(__VA_ARGS__); \
        case 128032: return bf ? FN<128, 32, __nv_bfloat16>(__VA_ARGS__) : FN<128, 32, float>(__VA_ARGS__); \
        case 128064: return bf ? FN<128, 64, __nv_bfloat16>(__VA_ARGS__) : FN<128, 64, float>(__VA_ARGS__); \
        case 128128: return bf ? FN<128, 128, __nv_bfloat16>(__VA_ARGS__) : FN<128, 128, float>(__VA_ARGS__); \
        default: return cudaErrorInvalidValue;                                        \
        }                                                                             \
    } while (0)

size_t simt_forward_workspace(int64_t BH, int64_t N, int d, int dv, int causal)
{
    if (N <= 0)
        return 0;
    const size_t E = (size_t)d * dv + d;
    size_t n = (size_t)BH * blocks_per_seq(N) * E;
    if (!causal)
        n += (size_t)BH * E;
    return n * sizeof(float);
}

size_t simt_state_workspace(int64_t BH, int64_t N, int d, int dv)
{
    return simt_forward_workspace(BH, N, d, dv, 1);
}

cudaError_t simt_forward(const FwdArgs& a) { LA_DISPATCH_DIMS(run_forward, a, false); }

cudaError_t simt_state(const FwdArgs& a) { LA_DISPATCH_DIMS(run_forward, a, true); }

}  // namespace la
