// la_decode.cu -- batched single-token decode step.
//
// One iteration of the causal recurrence on a stored state, for every
// sequence at once ("Efficient Attention Variants", sections 1 and 5: decode
// reads a fixed-shape state instead of a growing KV cache; "Linear Attention
// and SSM", eq. attn-linssm-recurrence):
//
//   S <- gamma S + phi(k) v^T,  z <- gamma z + phi(k),
//   o  = phi(q)^T S / max(phi(q)^T z, FLT_MIN)      (o = phi(q)^T S unnormalised)
//
// or, with a per-key-channel decay alpha (GLA, "Efficient Attention Variants"
// section 7.2), row i of S and entry i of z decay by alpha_i instead of gamma.
//
// The step is pure streaming: every state element is read once and written
// once (8 bytes per element), so the kernel is bound by HBM bandwidth.  One
// CTA owns one sequence's d x dv state; each thread keeps its RI rows of one
// 16-byte column group in registers, issues all of its loads before the first
// store, and writes back with streaming (evict-first) stores.  The read
// phi(q)^T S is reduced across the CTA through shared memory.
#include <float.h>

#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kThreads = 256;

template <int D, int DV>
struct DecodeTile {
    static constexpr int TJ = DV / 4;            // threads along value channels
    static constexpr int TI = kThreads / TJ;     // thread rows
    static constexpr int RI = D / TI;            // state rows per thread
    static_assert(D % TI == 0 && TJ <= kThreads, "tile");
};

// ALPHA: per-key-channel decay (GLA); else one gamma per head
template <int D, int DV, typename T, bool ALPHA>
__global__ void __launch_bounds__(kThreads)
    k_decode_step(float* __restrict__ S, float* __restrict__ z, const T* __restrict__ q,
                  const T* __restrict__ k, const T* __restrict__ v,
                  const float* __restrict__ alpha, float* __restrict__ out, int H, int fm,
                  GammaTable g)
{
    using TL = DecodeTile<D, DV>;
    __shared__ float sfq[D];
    __shared__ float sfk[D];
    __shared__ float sal[D];  // per-row decay of this step
    __shared__ __align__(16) float sv[DV];
    __shared__ __align__(16) float4 red[kThreads];
    __shared__ float sden[D / 32];

    const int64_t seq = blockIdx.x;
    const int head = (int)(seq % H);
    const int tid = threadIdx.x;
    const float gm = gamma_one(g, head);
    float* Sb = S + seq * (int64_t)(D * DV);
    const int tj = tid % TL::TJ, ti = tid / TL::TJ;

    // issue the state loads first: they are the whole cost of the step
    float4 s[TL::RI];
#pragma unroll
    for (int a = 0; a < TL::RI; ++a)
        s[a] = __ldcs(reinterpret_cast<const float4*>(Sb + (ti + a * TL::TI) * DV + tj * 4));

    if (tid < D) {
        sfq[tid] = phi_f32(to_f32<T>(q[seq * D + tid]), fm);
        sfk[tid] = phi_f32(to_f32<T>(k[seq * D + tid]), fm);
        if (ALPHA)
            sal[tid] = alpha[seq * D + tid];
    }
    if (tid < DV)
        sv[tid] = to_f32<T>(v[seq * DV + tid]);
    __syncthreads();

    // z update and phi(q).z on the first D threads (whole warps)
    if (tid < D) {
        float* zp = z + seq * D + tid;
        const float zn = fmaf(ALPHA ? sal[tid] : gm, *zp, sfk[tid]);
        *zp = zn;
        float part = sfq[tid] * zn;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            part += __shfl_xor_sync(0xffffffffu, part, o);
        if ((tid & 31) == 0)
            sden[tid >> 5] = part;
    }

    const float4 vv = *reinterpret_cast<const float4*>(sv + tj * 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int a = 0; a < TL::RI; ++a) {
        const int i = ti + a * TL::TI;
        const float f = sfk[i], ga = ALPHA ? sal[i] : gm;
        float4 x = s[a];
        x.x = fmaf(ga, x.x, f * vv.x);
        x.y = fmaf(ga, x.y, f * vv.y);
        x.z = fmaf(ga, x.z, f * vv.z);
        x.w = fmaf(ga, x.w, f * vv.w);
        __stcs(reinterpret_cast<float4*>(Sb + i * DV + tj * 4), x);
        const float fq = sfq[i];
        acc.x = fmaf(fq, x.x, acc.x);
        acc.y = fmaf(fq, x.y, acc.y);
        acc.z = fmaf(fq, x.z, acc.z);
        acc.w = fmaf(fq, x.w, acc.w);
    }
    red[tid] = acc;
    __syncthreads();
    if (tid < TL::TJ) {
        float4 r = red[tid];
        for (int m = 1; m < TL::TI; ++m) {
            const float4 y = red[tid + m * TL::TJ];
            r.x += y.x, r.y += y.y, r.z += y.z, r.w += y.w;
        }
        if (fm_normalised(fm)) {
            float den = 0.f;
#pragma unroll
            for (int w = 0; w < D / 32; ++w)
                den += sden[w];
            const float inv = 1.0f / fmaxf(den, FLT_MIN);
            r.x *= inv, r.y *= inv, r.z *= inv, r.w *= inv;
        }
        __stcs(reinterpret_cast<float4*>(out + seq * DV + tid * 4), r);
    }
}

template <int D, int DV, typename T>
cudaError_t run_decode(const DecodeArgs& a)
{
    auto kern = a.alpha ? k_decode_step<D, DV, T, true> : k_decode_step<D, DV, T, false>;
    kern<<<(unsigned)a.BH, kThreads, 0, a.stream>>>(
        a.S, a.z, static_cast<const T*>(a.q), static_cast<const T*>(a.k),
        static_cast<const T*>(a.v), a.alpha, a.out, (int)a.H, a.fm, *a.gamma);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t decode_step(const DecodeArgs& a)
{
    const bool bf = a.dtype == LA_BF16;
#define LA_DEC_CASE(D_, DV_)                                                         \
    case D_ * 1000 + DV_:                                                            \
        return bf ? run_decode<D_, DV_, __nv_bfloat16>(a) : run_decode<D_, DV_, float>(a);
    switch (a.d * 1000 + a.dv) {
        LA_DEC_CASE(32, 32)
        LA_DEC_CASE(32, 64)
        LA_DEC_CASE(32, 128)
        LA_DEC_CASE(64, 32)
        LA_DEC_CASE(64, 64)
        LA_DEC_CASE(64, 128)
        LA_DEC_CASE(128, 32)
        LA_DEC_CASE(128, 64)
        LA_DEC_CASE(128, 128)
    default:
        return cudaErrorInvalidValue;
    }
#undef LA_DEC_CASE
}

}  // namespace la
