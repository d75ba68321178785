// la_lasp.cu -- combining per-segment states for a sequence split (LASP-2).
//
// When a sequence is split into P consecutive parts (one per rank), part p
// summarises its own tokens as U_p (its final state from a zero start,
// la_state).  After an all-gather of the fixed-size U_p, the state before
// part `upto` is the exclusive prefix
//
//   P_0 = 0,   P_{p+1} = gamma^(len_p) P_p + U_p
//
// ("Linear Attention and SSM", LASP-2 section: one gather of fixed-size
// states, then a local prefix, independent of the sequence length;
// "Efficient Attention Variants", section 7.1: gamma^n weights a record n
// tokens old).  The rank then runs la_forward_with_state from P_upto.  One
// thread per state element, the parts in order.
#include <math.h>

#include "la_internal.cuh"

namespace la {
namespace {

constexpr int kMaxParts = 256;

struct PrefixParams {
    const float* S;  // [P][BH][d][dv]
    const float* z;  // [P][BH][d]
    float* S_out;    // [BH][d][dv]
    float* z_out;    // [BH][d]
    int64_t BH;
    int H, d, dv, upto;
    int64_t len[kMaxParts];
    GammaTable g;
};

__global__ void __launch_bounds__(256) k_state_prefix(const __grid_constant__ PrefixParams p)
{
    const int64_t E = (int64_t)p.d * p.dv + p.d;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.BH * E)
        return;
    const int64_t s = i / E, e = i % E;
    const int head = (int)(s % p.H);
    const bool zpart = e >= (int64_t)p.d * p.dv;
    const int64_t sz = p.BH * (int64_t)p.d * p.dv, zz = p.BH * (int64_t)p.d;
    const int64_t off = zpart ? s * p.d + (e - (int64_t)p.d * p.dv) : s * (int64_t)p.d * p.dv + e;
    float acc = 0.f;
    for (int q = 0; q < p.upto; ++q) {
        const float dec = p.g.has_decay ? exp2f((float)p.len[q] * p.g.log2g[head]) : 1.0f;
        const float u = zpart ? p.z[q * zz + off] : p.S[q * sz + off];
        acc = fmaf(dec, acc, u);
    }
    if (zpart)
        p.z_out[off] = acc;
    else
        p.S_out[off] = acc;
}

}  // namespace

int state_prefix_max_parts() { return kMaxParts; }

cudaError_t state_prefix(const float* S, const float* z, int nparts, const int64_t* len, int upto,
                         float* S_out, float* z_out, int64_t BH, int H, int d, int dv,
                         const GammaTable& g, cudaStream_t st)
{
    PrefixParams p;
    p.S = S, p.z = z, p.S_out = S_out, p.z_out = z_out;
    p.BH = BH, p.H = H, p.d = d, p.dv = dv, p.upto = upto;
    for (int q = 0; q < kMaxParts; ++q)
        p.len[q] = q < nparts ? len[q] : 0;
    p.g = g;
    const int64_t n = BH * ((int64_t)d * dv + d);
    k_state_prefix<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace la
