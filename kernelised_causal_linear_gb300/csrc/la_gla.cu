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
// Chunked in three launches like the scalar-decay path, in fp32, with every
// decay factor taken as exp of a difference of running log-sums, so that no
// factor exceeds 1 (no ratio of small products); with bf16 inputs at d = 128
// the products of steps 1 and 3 run on the tensor cores (warp-level bf16
// MMAs with fp32 accumulation, fp32 operands as bf16 hi/lo pairs):
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

// Warp-level bf16 tensor-core products (mma.sync m16n8k16, fp32
// accumulate) for the sub-chunk products of the block-state and output
// kernels with bf16 inputs.  Fragment layouts (lane = 4 g + q): A 16 x 16 row-major, registers
// {A[g][2q..2q+1]}, {A[g+8][2q..]}, {A[g][2q+8..]}, {A[g+8][2q+8..]}; B 16 x 8,
// {B[2q..2q+1][g]}, {B[2q+8..2q+9][g]}; C 16 x 8, C[g][2q], C[g][2q+1],
// C[g+8][2q], C[g+8][2q+1].
__device__ __forceinline__ uint32_t bf2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// two fp32 -> packed bf16 hi and lo parts (hi + lo = x to ~2^-17)
__device__ __forceinline__ void bf2_split(float a, float b, uint32_t& hi, uint32_t& lo)
{
    hi = bf2(a, b);
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&hi);
    lo = bf2(a - __low2float(h), b - __high2float(h));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A[m][k] = X[k * ld + m] (X stored transposed), tile rows m0.., k0.., as hi and lo
// parts
__device__ __forceinline__ void frag_a_t_split(const float* X, int ld, int m0, int k0, int g,
                                               int q, uint32_t (&ah)[4], uint32_t (&al)[4])
{
    const float* p = X + (k0 + 2 * q) * ld + m0 + g;
    bf2_split(p[0], p[ld], ah[0], al[0]);
    bf2_split(p[8], p[ld + 8], ah[1], al[1]);
    bf2_split(p[8 * ld], p[9 * ld], ah[2], al[2]);
    bf2_split(p[8 * ld + 8], p[9 * ld + 8], ah[3], al[3]);
}

// A[m][k] from packed pairs along k: word (k / 2) * ld + m holds
// (A[m][k], A[m][k + 1]) (k even)
__device__ __forceinline__ void frag_a_p(const uint32_t* P, int ld, int m0, int k0, int g, int q,
                                         uint32_t (&a)[4])
{
    const uint32_t* p = P + (k0 / 2 + q) * ld + m0 + g;
    a[0] = p[0];
    a[1] = p[8];
    a[2] = p[4 * ld];
    a[3] = p[4 * ld + 8];
}

// A[m][k] = X[m * ld + k] (row-major, ld and k0 even), as hi and lo parts
__device__ __forceinline__ void frag_a_r_split(const float* X, int ld, int m0, int k0, int g, int q,
                                               uint32_t (&ah)[4], uint32_t (&al)[4])
{
    const float* p = X + (m0 + g) * ld + k0 + 2 * q;
    const float2 x0 = *reinterpret_cast<const float2*>(p);
    const float2 x1 = *reinterpret_cast<const float2*>(p + 8 * ld);
    const float2 x2 = *reinterpret_cast<const float2*>(p + 8);
    const float2 x3 = *reinterpret_cast<const float2*>(p + 8 * ld + 8);
    bf2_split(x0.x, x0.y, ah[0], al[0]);
    bf2_split(x1.x, x1.y, ah[1], al[1]);
    bf2_split(x2.x, x2.y, ah[2], al[2]);
    bf2_split(x3.x, x3.y, ah[3], al[3]);
}

// B[k][n] = X[k * ld + n], tile k0.., n0..
__device__ __forceinline__ void frag_b(const float* X, int ld, int k0, int n0, int g, int q,
                                       uint32_t& b0, uint32_t& b1)
{
    const float* p = X + (k0 + 2 * q) * ld + n0 + g;
    b0 = bf2(p[0], p[ld]);
    b1 = bf2(p[8 * ld], p[9 * ld]);
}

__device__ __forceinline__ void frag_b_split(const float* X, int ld, int k0, int n0, int g, int q,
                                             uint32_t (&bh)[2], uint32_t (&bl)[2])
{
    const float* p = X + (k0 + 2 * q) * ld + n0 + g;
    bf2_split(p[0], p[ld], bh[0], bl[0]);
    bf2_split(p[8 * ld], p[9 * ld], bh[1], bl[1]);
}

// ------------------------------------------------------------- step 1 ----
// Thread (ti, tj) owns RI consecutive rows (channels) x RJ consecutive value
// columns of the D x DV block state: per token, RI + RJ shared loads (16-byte
// where they line up) feed RI x RJ FMAs.  The running log-sum of each channel
// is kept by thread i < D.
template <int D, int DV>
struct StateTile {
    static constexpr int RJ = (D * DV / kThreads >= 8) ? 8 : 4;
    static constexpr int TJ = DV / RJ;
    static constexpr int TI = kThreads / TJ;
    static constexpr int RI = D / TI;
    static_assert(RI >= 1 && TI * TJ == kThreads && RI * TI == D, "state tile");
};

template <int N>
__device__ __forceinline__ void lds_row(const float* p, float (&x)[N])
{
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const float4 v = reinterpret_cast<const float4*>(p)[q];
            x[4 * q] = v.x, x[4 * q + 1] = v.y, x[4 * q + 2] = v.z, x[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < N; ++q)
            x[q] = p[q];
    }
}

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kThreads)
    k_gla_state(const T* __restrict__ kp, const T* __restrict__ vp, const float* __restrict__ ap,
                float* __restrict__ ws, float* __restrict__ dec, int64_t N, int nblk, int fm)
{
    using TL = StateTile<D, DV>;
    constexpr int TJ = TL::TJ, RI = TL::RI, RJ = TL::RJ;
    // bf16 inputs at d = 128: each sub-chunk's part of the block state is a
    // tensor-core product (mma.sync m16n8k16, fp32 accumulation) of the
    // weighted phi(k), an fp32 bf16 hi/lo pair, and v, exact in bf16; warp w
    // owns state rows 16 w .. 16 w + 15 (the log gates use the hardware
    // logarithm, as in the output kernel)
    constexpr bool kMma = sizeof(T) == 2 && D == 128 && (DV == 128 || DV == 64);
    constexpr int NT = DV / 8;  // 8-column tiles of a warp's rows
    // dynamic shared memory (more than the 48 KiB of static arrays with
    // D = DV = 128): phi(k) o exp(L_e - L_t) with L_e the sub-chunk's last
    // L, v (rows padded by 4 floats, so that the operand fragments hit
    // different banks), log alpha, the sub-chunk's decay exp(L_e - L_s)
    // per channel (L_s: L before the sub-chunk)
    extern __shared__ __align__(16) float st_smem[];
    float(*sk)[D + 4] = reinterpret_cast<float(*)[D + 4]>(st_smem);
    float(*sv)[DV + 4] = reinterpret_cast<float(*)[DV + 4]>(st_smem + kSub * (D + 4));
    // the tensor-core form keeps v as bf16 pairs of consecutive tokens, word
    // (t / 2) * (DV + 8) + c, in the same space
    __nv_bfloat16* v2h = reinterpret_cast<__nv_bfloat16*>(&sv[0][0]);
    const uint32_t* v2w = reinterpret_cast<const uint32_t*>(&sv[0][0]);
    float(*sl)[D] = reinterpret_cast<float(*)[D]>(st_smem + kSub * (D + DV + 8));
    float* sdec = st_smem + kSub * (2 * D + DV + 8);
    float* sle = sdec + D;  // L_e per channel
    const int64_t gb = blockIdx.x;
    const int64_t seq = gb / nblk;
    const int blk = (int)(gb % nblk);
    const int64_t t0 = (int64_t)blk * kBlockL;
    const int len = (int)min((int64_t)kBlockL, N - t0);
    const T* kb = kp + (seq * N + t0) * D;
    const T* vb = vp + (seq * N + t0) * DV;
    const float* ab = ap + (seq * N + t0) * D;
    const int tid = threadIdx.x, tj = tid % TJ, ti = tid / TJ;

    // The state so far is kept relative to the end of the tokens folded in:
    // before each sub-chunk it decays by the sub-chunk's exp(L_e - L_s) per
    // channel, and the sub-chunk's tokens enter with exp(L_e - L_t), so that
    // the last token of the block has weight exactly 1 and no pass over the
    // block's gates is needed before the first sub-chunk.
    float run = 0.f;  // L_t of channel tid (tid < D), running
    float acc[RI][RJ];
#pragma unroll
    for (int a = 0; a < RI; ++a)
#pragma unroll
        for (int b = 0; b < RJ; ++b)
            acc[a][b] = 0.f;
    float macc[kMma ? NT : 1][4];
#pragma unroll
    for (int nt = 0; nt < (kMma ? NT : 1); ++nt)
        macc[nt][0] = macc[nt][1] = macc[nt][2] = macc[nt][3] = 0.f;
    const int lane = tid & 31, warp = tid >> 5, g = lane >> 2, q = lane & 3;
    float zacc = 0.f;
    for (int s0 = 0; s0 < len; s0 += kSub) {
        const int n = min(kSub, len - s0);
        {
            // loads issued in batches of up to eight elements before use
            constexpr int NE = kSub * D / kThreads, NB = NE < 8 ? NE : 8;
#pragma unroll 1
            for (int x0 = 0; x0 < NE; x0 += NB) {
                float ra[NB], rk[NB];
#pragma unroll
                for (int x = 0; x < NB; ++x) {
                    const int e = tid + (x0 + x) * kThreads;
                    const int t = e / D, i = e % D;
                    ra[x] = 1.f, rk[x] = 0.f;
                    if (t < n) {
                        ra[x] = __ldg(ab + (int64_t)(s0 + t) * D + i);
                        rk[x] = ldf(kb + (int64_t)(s0 + t) * D + i);
                    }
                }
#pragma unroll
                for (int x = 0; x < NB; ++x) {
                    const int e = tid + (x0 + x) * kThreads;
                    const int t = e / D, i = e % D;
                    const bool in = t < n;
                    sl[t][i] = in ? (kMma ? __logf(ra[x]) : logf(ra[x])) : 0.f;
                    sk[t][i] = in ? phi_f32(rk[x], fm) : 0.f;
                }
            }
        }
        __syncthreads();
        if (tid < D) {  // the running log-sum
            const float start = run;
            for (int t = 0; t < n; ++t) {
                run += sl[t][tid];
                sl[t][tid] = run;
            }
            sdec[tid] = expf(run - start);
            sle[tid] = run;
        }
        {
            constexpr int NVE = kSub * DV / kThreads, NB = NVE < 8 ? NVE : 8;
#pragma unroll 1
            for (int x0 = 0; x0 < NVE; x0 += NB) {
                float rv[NB];
#pragma unroll
                for (int x = 0; x < NB; ++x) {
                    const int e = tid + (x0 + x) * kThreads;
                    const int t = e / DV, c = e % DV;
                    rv[x] = t < n ? ldf(vb + (int64_t)(s0 + t) * DV + c) : 0.f;
                }
#pragma unroll
                for (int x = 0; x < NB; ++x) {
                    const int e = tid + (x0 + x) * kThreads;
                    if constexpr (kMma)  // bf16 pairs of consecutive tokens (exact)
                        v2h[((e / DV) >> 1) * (2 * (DV + 8)) + 2 * (e % DV) + ((e / DV) & 1)] =
                            __float2bfloat16_rn(rv[x]);
                    else
                        sv[e / DV][e % DV] = rv[x];
                }
            }
        }
        __syncthreads();
        // the weights exp(L_e - L_t), spread over every thread
        for (int e = tid; e < n * D; e += kThreads) {
            const int t = e / D, i = e % D;
            sk[t][i] *= expf(sle[i] - sl[t][i]);
        }
        __syncthreads();
        if constexpr (kMma) {
            {
                const float f0 = sdec[16 * warp + g], f1 = sdec[16 * warp + g + 8];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    macc[nt][0] *= f0, macc[nt][1] *= f0;
                    macc[nt][2] *= f1, macc[nt][3] *= f1;
                }
            }
#pragma unroll
            for (int k0 = 0; k0 < kSub; k0 += 16) {
                uint32_t ah[4], al[4];
                frag_a_t_split(&sk[0][0], D + 4, 16 * warp, k0, g, q, ah, al);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t b0 = v2w[(k0 / 2 + q) * (DV + 8) + 8 * nt + g];
                    const uint32_t b1 = v2w[(k0 / 2 + q + 4) * (DV + 8) + 8 * nt + g];
                    mma16816(macc[nt], ah, b0, b1);
                    mma16816(macc[nt], al, b0, b1);
                }
            }
            if (tid < D) {
                zacc *= sdec[tid];
                for (int t = 0; t < kSub; ++t)
                    zacc += sk[t][tid];
            }
        } else {
#pragma unroll
            for (int a = 0; a < RI; ++a) {
                const float f = sdec[ti * RI + a];
#pragma unroll
                for (int b = 0; b < RJ; ++b)
                    acc[a][b] *= f;
            }
            if (tid < D)
                zacc *= sdec[tid];
#pragma unroll 4
            for (int t = 0; t < kSub; ++t) {
                float kr[RI], vr[RJ];
                lds_row(&sk[t][ti * RI], kr);
                lds_row(&sv[t][tj * RJ], vr);
#pragma unroll
                for (int a = 0; a < RI; ++a)
#pragma unroll
                    for (int b = 0; b < RJ; ++b)
                        acc[a][b] = fmaf(kr[a], vr[b], acc[a][b]);
                if (tid < D)
                    zacc += sk[t][tid];
            }
        }
        __syncthreads();
    }
    float* dst = ws + gb * (int64_t)(D * DV + D);
    if constexpr (kMma) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int i = 16 * warp + g, c = 8 * nt + 2 * q;
            *reinterpret_cast<float2*>(dst + i * DV + c) = make_float2(macc[nt][0], macc[nt][1]);
            *reinterpret_cast<float2*>(dst + (i + 8) * DV + c) = make_float2(macc[nt][2], macc[nt][3]);
        }
    } else {
#pragma unroll
        for (int a = 0; a < RI; ++a) {
            const int i = ti * RI + a;
#pragma unroll
            for (int qq = 0; qq < RJ / 4; ++qq)
                *reinterpret_cast<float4*>(dst + i * DV + tj * RJ + 4 * qq) =
                    make_float4(acc[a][4 * qq], acc[a][4 * qq + 1], acc[a][4 * qq + 2],
                                acc[a][4 * qq + 3]);
        }
    }
    if (tid < D) {
        dst[D * DV + tid] = zacc;
        dec[gb * D + tid] = expf(run);
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
    // kAhead blocks' values and decays in flight at a time
    constexpr int kAhead = 8;
    float acc = 0.f;
    for (int b0 = 0; b0 < nblk; b0 += kAhead) {
        float x[kAhead], dd[kAhead];
#pragma unroll
        for (int i = 0; i < kAhead; ++i)
            if (b0 + i < nblk) {
                x[i] = __ldcg(base + (int64_t)(b0 + i) * E);
                dd[i] = __ldg(db + (int64_t)(b0 + i) * D);
            }
#pragma unroll
        for (int i = 0; i < kAhead; ++i)
            if (b0 + i < nblk) {
                base[(int64_t)(b0 + i) * E] = acc;
                acc = fmaf(acc, dd[i], x[i]);
            }
    }
}

// ------------------------------------------------------------- step 3 ----
// Shared memory of the output kernel (floats): the running state S [D][DV]
// and z [D]; phi(q), phi(k) and the running log-sums L of the sub-chunk,
// transposed ([D][LDT], token fastest); v [kSub][DV]; the intra weights
// transposed (AT[j][t]); the denominators.
template <int D, int DV>
struct GlaOut {
    static constexpr int LDT = kSub + 4;
    // row strides of the state and value tiles: 4 floats of padding put
    // rows 2q (q = 0..3) of a tensor-core operand fragment in different banks
    static constexpr int SS = DV + 4, SV = DV + 4;
    static constexpr size_t oZ = (size_t)D * SS, oQ = oZ + D, oK = oQ + (size_t)D * LDT,
                            oL = oK + (size_t)D * LDT, oV = oL + (size_t)D * LDT,
                            oA = oV + (size_t)kSub * SV, oDen = oA + (size_t)kSub * LDT,
                            floats = oDen + kSub;
    static constexpr size_t bytes = floats * sizeof(float);
    // output tiles of 4 tokens x 4 value columns (OT threads); state-update
    // tiles of UR channels x 8 value columns (UT threads)
    static constexpr int OJ = DV / 4, OI = kSub / 4, OT = OI * OJ;
    static constexpr int UR = D * DV / 8 >= 4 * kThreads ? 4 : D * DV / 8 >= 2 * kThreads ? 2 : 1;
    static constexpr int UJ = DV / 8, UI = D / UR, UT = UI * UJ;
    static_assert(OT <= kThreads && UT <= kThreads && DV % 8 == 0, "tiles");
};

template <int D, int DV, typename T>
__global__ void __launch_bounds__(kThreads, 2)
    k_gla_out(const T* __restrict__ qp, const T* __restrict__ kp, const T* __restrict__ vp,
              const float* __restrict__ ap, float* __restrict__ out, const float* __restrict__ ws,
              int64_t N, int nblk, int fm)
{
    // a CTA takes DVC of the DV value columns (two CTAs per block with
    // DV = 128: half the state in shared memory, two CTAs per SM)
    constexpr int DVC = DV > 64 ? 64 : DV, NH = DV / DVC;
    using G = GlaOut<D, DVC>;
    constexpr int LDT = G::LDT, SS = G::SS, SV = G::SV, E = D * DV + D;
    // bf16 inputs at d = 128 with 64 value columns per CTA: the products of
    // a sub-chunk whose decay factors split run on the tensor cores (bf16
    // operands, fp32 accumulation).  The rescaled features, the state and the
    // intra weights are fp32 and enter as bf16 hi/lo pairs (hi*hi + hi*lo +
    // lo*hi, ~2^-16 relative: a single rounding of the features showed in
    // the unnormalised outputs, whose sums cancel); v is exact in bf16.  The
    // log gates use the hardware logarithm (absolute error below 2^-21 on
    // [0.5, 2], three ulp elsewhere), far inside the bf16 tolerance.
    constexpr bool kMma = sizeof(T) == 2 && D == 128 && DVC == 64;
    extern __shared__ __align__(16) float smem[];
    float* sS = smem;
    float* sz = smem + G::oZ;
    float* qT = smem + G::oQ;  // qT[i * LDT + t]
    float* kT = smem + G::oK;
    float* LT = smem + G::oL;
    float* sv = smem + G::oV;  // sv[t * SV + c]
    float* AT = smem + G::oA;  // AT[j * LDT + t]
    float* sden = smem + G::oDen;

    const int64_t gb = blockIdx.x / NH;
    const int c_off = (int)(blockIdx.x % NH) * DVC;
    const int64_t seq = gb / nblk;
    const int blk = (int)(gb % nblk);
    const int64_t t0 = (int64_t)blk * kBlockL;
    const int len = (int)min((int64_t)kBlockL, N - t0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool norm = fm_normalised(fm);
    for (int e = tid; e < D * DVC; e += kThreads)
        sS[(e / DVC) * SS + e % DVC] = ws[gb * E + (e / DVC) * DV + c_off + e % DVC];
    for (int i = tid; i < D; i += kThreads)
        sz[i] = ws[gb * E + D * DV + i];
    const T* qb = qp + (seq * N + t0) * D;
    const T* kb = kp + (seq * N + t0) * D;
    const T* vb = vp + (seq * N + t0) * DV + c_off;
    const float* ab = ap + (seq * N + t0) * D;
    float* ob = out + (seq * N + t0) * DV + c_off;

    for (int s0 = 0; s0 < len; s0 += kSub) {
        const int n = min(kSub, len - s0);
        __syncthreads();  // the previous sub-chunk is consumed
        // log alpha, phi(q), phi(k) of the sub-chunk (coalesced, every thread),
        // then channel tid < D turns its log alphas into the running sum L
        // (a warp takes 8 channels x 4 tokens: the transposed stores hit 32
        // different banks)
        // (all of a thread's loads are issued before any is used: the
        // staging is bound by global-load latency otherwise)
        {
            constexpr int NE = kSub * D / kThreads, NVE = kSub * DVC / kThreads;
            float ra[NE], rq[NE], rk[NE], rv[NVE];
#pragma unroll
            for (int x = 0; x < NE; ++x) {
                const int e = tid + x * kThreads;
                const int wt = e >> 5, cg = wt % (D / 8), tg = wt / (D / 8);
                const int i = 8 * cg + (e & 7), t = 4 * tg + ((e >> 3) & 3);
                ra[x] = 1.f, rq[x] = 0.f, rk[x] = 0.f;
                if (t < n) {
                    const int64_t o = (int64_t)(s0 + t) * D + i;
                    ra[x] = __ldg(ab + o);
                    rq[x] = ldf(qb + o);
                    rk[x] = ldf(kb + o);
                }
            }
#pragma unroll
            for (int x = 0; x < NVE; ++x) {
                const int e = tid + x * kThreads;
                const int t = e / DVC, c = e % DVC;
                rv[x] = t < n ? ldf(vb + (int64_t)(s0 + t) * DV + c) : 0.f;
            }
#pragma unroll
            for (int x = 0; x < NE; ++x) {
                const int e = tid + x * kThreads;
                const int wt = e >> 5, cg = wt % (D / 8), tg = wt / (D / 8);
                const int i = 8 * cg + (e & 7), t = 4 * tg + ((e >> 3) & 3);
                const bool in = t < n;
                LT[i * LDT + t] = in ? (kMma ? __logf(ra[x]) : logf(ra[x])) : 0.f;
                qT[i * LDT + t] = in ? phi_f32(rq[x], fm) : 0.f;
                kT[i * LDT + t] = in ? phi_f32(rk[x], fm) : 0.f;
            }
#pragma unroll
            for (int x = 0; x < NVE; ++x)
                sv[((tid + x * kThreads) / DVC) * SV + (tid + x * kThreads) % DVC] = rv[x];
        }
        __syncthreads();
        if (tid < D) {  // channel tid's 32 log gates in registers, summed in token order
            float4* row = reinterpret_cast<float4*>(LT + tid * LDT);
            float4 x[kSub / 4];
#pragma unroll
            for (int u = 0; u < kSub / 4; ++u)
                x[u] = row[u];
            float run = 0.f;
#pragma unroll
            for (int u = 0; u < kSub / 4; ++u) {
                run += x[u].x, x[u].x = run;
                run += x[u].y, x[u].y = run;
                run += x[u].z, x[u].z = run;
                run += x[u].w, x[u].w = run;
            }
#pragma unroll
            for (int u = 0; u < kSub / 4; ++u)
                row[u] = x[u];
        }
        // When the sub-chunk's decay stays above e^-60 in every channel,
        // exp(L_t - L_j) = exp(L_t) exp(-L_j) with both factors in fp32 range:
        // phi(q) and phi(k) are rescaled once and every product below is a
        // plain sum of products; otherwise each factor is taken as exp of a
        // difference.  (Thread tid < D tests its own channel, written above
        // by itself.)
        const bool split =
            __syncthreads_and(tid >= D || LT[tid * LDT + n - 1] >= -60.0f) != 0;
        // tensor-core form: phi(q) o exp(L_t) as bf16 hi and lo parts of pairs
        // of consecutive channels, word (i / 2) * LDT + t of the hi plane and
        // the same word of the lo plane after it, in place of qT (the
        // fragments of every warp then load words instead of splitting)
        uint32_t* q2 = reinterpret_cast<uint32_t*>(qT);
        const uint32_t* q2h = q2;
        const uint32_t* q2l = q2 + (D / 2) * LDT;
        if (kMma && split) {
            // every thread rescales pairs of channels at one token, packs
            // phi(q) in registers, and writes the planes once every read of
            // the fp32 tile is done
            constexpr int NP = (D / 2) * kSub / kThreads;
            uint32_t ph[NP], pl[NP];
#pragma unroll
            for (int x = 0; x < NP; ++x) {
                const int e = tid + x * kThreads, ip = e / kSub, t = e % kSub;
                const int o0 = 2 * ip * LDT + t, o1 = o0 + LDT;
                const float l0 = LT[o0], l1 = LT[o1];
                bf2_split(qT[o0] * expf(l0), qT[o1] * expf(l1), ph[x], pl[x]);
                kT[o0] *= expf(-l0);
                kT[o1] *= expf(-l1);
            }
            __syncthreads();
#pragma unroll
            for (int x = 0; x < NP; ++x) {
                const int e = tid + x * kThreads, ip = e / kSub, t = e % kSub;
                q2[ip * LDT + t] = ph[x];
                q2[(D / 2) * LDT + ip * LDT + t] = pl[x];
            }
            __syncthreads();
        } else if (split) {
            if (tid < D)
                for (int t = 0; t < kSub; ++t) {
                    const float l = LT[tid * LDT + t];
                    qT[tid * LDT + t] *= expf(l);
                    kT[tid * LDT + t] *= expf(-l);
                }
            __syncthreads();
        }
        // intra weights A_tj = sum_i q_ti k_ji exp(L_ti - L_ji), j <= t:
        // thread (ty, tx) takes tokens 4 ty .. 4 ty + 3 and key token tx
        if (kMma && split) {
            // warp w: tokens 16 (w & 1) .. + 15, keys 8 (w >> 1) .. + 7
            const int g = lane >> 2, q = lane & 3, m0 = 16 * (warp & 1), n0 = 8 * (warp >> 1);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k0 = 0; k0 < D; k0 += 16) {
                uint32_t ah[4], al[4], bh[2], bl[2];
                frag_a_p(q2h, LDT, m0, k0, g, q, ah);
                frag_a_p(q2l, LDT, m0, k0, g, q, al);
                frag_b_split(kT, LDT, k0, n0, g, q, bh, bl);
                mma16816(acc, ah, bh[0], bh[1]);
                mma16816(acc, ah, bl[0], bl[1]);
                mma16816(acc, al, bh[0], bh[1]);
            }
            const int t0 = m0 + g, j0 = n0 + 2 * q;
            AT[j0 * LDT + t0] = j0 <= t0 ? acc[0] : 0.f;
            AT[(j0 + 1) * LDT + t0] = j0 + 1 <= t0 ? acc[1] : 0.f;
            AT[j0 * LDT + t0 + 8] = j0 <= t0 + 8 ? acc[2] : 0.f;
            AT[(j0 + 1) * LDT + t0 + 8] = j0 + 1 <= t0 + 8 ? acc[3] : 0.f;
        } else if (split) {
            // 64 threads, 4 tokens x 4 key tokens each (two 16-byte loads per
            // 16 FMAs)
            if (tid < (kSub / 4) * (kSub / 4)) {
                const int ty = tid / (kSub / 4), jx = tid % (kSub / 4);
                float acc[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
#pragma unroll 8
                for (int i = 0; i < D; ++i) {
                    const float4 q4 = *reinterpret_cast<const float4*>(qT + i * LDT + 4 * ty);
                    const float4 k4 = *reinterpret_cast<const float4*>(kT + i * LDT + 4 * jx);
                    const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        acc[r][0] = fmaf(qv[r], k4.x, acc[r][0]);
                        acc[r][1] = fmaf(qv[r], k4.y, acc[r][1]);
                        acc[r][2] = fmaf(qv[r], k4.z, acc[r][2]);
                        acc[r][3] = fmaf(qv[r], k4.w, acc[r][3]);
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = 4 * jx + c;
                    float w[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        w[r] = j <= 4 * ty + r ? acc[r][c] : 0.f;
                    *reinterpret_cast<float4*>(AT + j * LDT + 4 * ty) = make_float4(w[0], w[1], w[2], w[3]);
                }
            }
        } else {
            const int ty = tid >> 5, tx = lane;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            {
                for (int i = 0; i < D; ++i) {
                    const float kk = kT[i * LDT + tx], lj = LT[i * LDT + tx];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        acc[r] = fmaf(qT[i * LDT + 4 * ty + r] * kk,
                                      __expf(LT[i * LDT + 4 * ty + r] - lj), acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (tx > 4 * ty + r)
                    acc[r] = 0.f;
            *reinterpret_cast<float4*>(AT + tx * LDT + 4 * ty) =
                make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
        __syncthreads();
        // denominators: (phi(q_t) o exp(L_t)) . z + sum_j A_tj, one warp per
        // four tokens
        if (norm) {
            for (int t = 4 * warp; t < 4 * warp + 4; ++t) {
                float part = lane <= t ? AT[lane * LDT + t] : 0.f;
                for (int i = lane; i < D; i += 32) {
                    float qi;
                    if (kMma && split) {
                        const __nv_bfloat16* hh = reinterpret_cast<const __nv_bfloat16*>(q2h);
                        const __nv_bfloat16* ll = reinterpret_cast<const __nv_bfloat16*>(q2l);
                        const int w2 = 2 * ((i >> 1) * LDT + t) + (i & 1);
                        qi = __bfloat162float(hh[w2]) + __bfloat162float(ll[w2]);
                    } else {
                        qi = split ? qT[i * LDT + t] : qT[i * LDT + t] * expf(LT[i * LDT + t]);
                    }
                    part = fmaf(qi, sz[i], part);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    part += __shfl_xor_sync(0xffffffffu, part, o);
                if (lane == 0)
                    sden[t] = part;
            }
            __syncthreads();
        }
        // outputs: thread (oi, oj) < OT takes 4 tokens x 4 columns
        if (kMma && split) {
            // warp w: value columns 8 w .. 8 w + 7 of all 32 tokens
            const int g = lane >> 2, q = lane & 3, n0 = 8 * warp;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 2
            for (int k0 = 0; k0 < D; k0 += 16) {
                uint32_t bh[2], bl[2];
                frag_b_split(sS, SS, k0, n0, g, q, bh, bl);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    uint32_t ah[4], al[4];
                    frag_a_p(q2h, LDT, 16 * mt, k0, g, q, ah);
                    frag_a_p(q2l, LDT, 16 * mt, k0, g, q, al);
                    mma16816(acc[mt], ah, bh[0], bh[1]);
                    mma16816(acc[mt], ah, bl[0], bl[1]);
                    mma16816(acc[mt], al, bh[0], bh[1]);
                }
            }
#pragma unroll
            for (int k0 = 0; k0 < kSub; k0 += 16) {
                uint32_t b0, b1;
                frag_b(sv, SV, k0, n0, g, q, b0, b1);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    uint32_t ah[4], al[4];
                    frag_a_t_split(AT, LDT, 16 * mt, k0, g, q, ah, al);
                    mma16816(acc[mt], ah, b0, b1);
                    mma16816(acc[mt], al, b0, b1);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int t = 16 * mt + g + 8 * h;
                    if (t < n) {
                        float2 o = make_float2(acc[mt][2 * h], acc[mt][2 * h + 1]);
                        if (norm) {
                            const float inv = 1.0f / fmaxf(sden[t], FLT_MIN);
                            o.x *= inv, o.y *= inv;
                        }
                        *reinterpret_cast<float2*>(ob + (int64_t)(s0 + t) * DV + n0 + 2 * q) = o;
                    }
                }
        } else if (tid < G::OT) {
            constexpr int ORI = 4;
            const int oj = tid % G::OJ, oi = tid / G::OJ;
            const int tb = oi * ORI, c0 = 4 * oj;
            float acc[ORI][4];
#pragma unroll
            for (int r = 0; r < ORI; ++r)
                acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
#pragma unroll 4
            for (int i = 0; i < D; ++i) {
                float qv[ORI];
                lds_row(qT + i * LDT + tb, qv);
                if (!split)
#pragma unroll
                    for (int r = 0; r < ORI; ++r)
                        qv[r] *= expf(LT[i * LDT + tb + r]);
                const float4 s4 = *reinterpret_cast<const float4*>(sS + i * SS + c0);
#pragma unroll
                for (int r = 0; r < ORI; ++r) {
                    acc[r][0] = fmaf(qv[r], s4.x, acc[r][0]);
                    acc[r][1] = fmaf(qv[r], s4.y, acc[r][1]);
                    acc[r][2] = fmaf(qv[r], s4.z, acc[r][2]);
                    acc[r][3] = fmaf(qv[r], s4.w, acc[r][3]);
                }
            }
#pragma unroll 4
            for (int j = 0; j < kSub; ++j) {
                float av[ORI];
                lds_row(AT + j * LDT + tb, av);
                const float4 v4 = *reinterpret_cast<const float4*>(sv + j * SV + c0);
#pragma unroll
                for (int r = 0; r < ORI; ++r) {
                    acc[r][0] = fmaf(av[r], v4.x, acc[r][0]);
                    acc[r][1] = fmaf(av[r], v4.y, acc[r][1]);
                    acc[r][2] = fmaf(av[r], v4.z, acc[r][2]);
                    acc[r][3] = fmaf(av[r], v4.w, acc[r][3]);
                }
            }
#pragma unroll
            for (int r = 0; r < ORI; ++r) {
                const int t = tb + r;
                if (t < n) {
                    float4 o = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
                    if (norm) {
                        const float inv = 1.0f / fmaxf(sden[t], FLT_MIN);
                        o.x *= inv, o.y *= inv, o.z *= inv, o.w *= inv;
                    }
                    *reinterpret_cast<float4*>(ob + (int64_t)(s0 + t) * DV + c0) = o;
                }
            }
        }
        __syncthreads();  // every read of S, z for this sub-chunk is done
        // S <- diag(exp(L_end)) S + sum_j (phi(k_j) o exp(L_end - L_j)) v_j^T ; z alike
        if (kMma && split) {
            // warp w: channels 16 w .. 16 w + 15, all 64 value columns; the
            // accumulators start from S and end scaled by exp(L_end)
            const int g = lane >> 2, q = lane & 3, m0 = 16 * warp;
            float acc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const float2 x0 = *reinterpret_cast<const float2*>(sS + (m0 + g) * SS + 8 * nt + 2 * q);
                const float2 x1 =
                    *reinterpret_cast<const float2*>(sS + (m0 + g + 8) * SS + 8 * nt + 2 * q);
                acc[nt][0] = x0.x, acc[nt][1] = x0.y, acc[nt][2] = x1.x, acc[nt][3] = x1.y;
            }
#pragma unroll
            for (int k0 = 0; k0 < kSub; k0 += 16) {
                uint32_t ah[4], al[4];
                frag_a_r_split(kT, LDT, m0, k0, g, q, ah, al);
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    uint32_t b0, b1;
                    frag_b(sv, SV, k0, 8 * nt, g, q, b0, b1);
                    mma16816(acc[nt], ah, b0, b1);
                    mma16816(acc[nt], al, b0, b1);
                }
            }
            const float g0 = expf(LT[(m0 + g) * LDT + n - 1]), g1 = expf(LT[(m0 + g + 8) * LDT + n - 1]);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                *reinterpret_cast<float2*>(sS + (m0 + g) * SS + 8 * nt + 2 * q) =
                    make_float2(g0 * acc[nt][0], g0 * acc[nt][1]);
                *reinterpret_cast<float2*>(sS + (m0 + g + 8) * SS + 8 * nt + 2 * q) =
                    make_float2(g1 * acc[nt][2], g1 * acc[nt][3]);
            }
        } else if (tid < G::UT) {
            constexpr int RI = G::UR, RJ = 8;
            const int tj = tid % G::UJ, ti = tid / G::UJ;
            float g[RI], acc[RI][RJ];
#pragma unroll
            for (int a = 0; a < RI; ++a) {
                const int i = ti * RI + a;
                g[a] = expf(LT[i * LDT + n - 1]);
                float row[RJ];
                lds_row(sS + i * SS + tj * RJ, row);
#pragma unroll
                for (int b = 0; b < RJ; ++b)
                    acc[a][b] = split ? row[b] : g[a] * row[b];
            }
#pragma unroll 4
            for (int j = 0; j < kSub; ++j) {
                float kr[RI], vr[RJ];
#pragma unroll
                for (int a = 0; a < RI; ++a) {
                    const int i = ti * RI + a;
                    kr[a] = split ? kT[i * LDT + j]
                                  : kT[i * LDT + j] * __expf(LT[i * LDT + n - 1] - LT[i * LDT + j]);
                }
                lds_row(sv + j * SV + tj * RJ, vr);
#pragma unroll
                for (int a = 0; a < RI; ++a)
#pragma unroll
                    for (int b = 0; b < RJ; ++b)
                        acc[a][b] = fmaf(kr[a], vr[b], acc[a][b]);
            }
#pragma unroll
            for (int a = 0; a < RI; ++a) {
                const int i = ti * RI + a;
#pragma unroll
                for (int q = 0; q < RJ / 4; ++q) {
                    const float m = split ? g[a] : 1.0f;
                    *reinterpret_cast<float4*>(sS + i * SS + tj * RJ + 4 * q) =
                        make_float4(m * acc[a][4 * q], m * acc[a][4 * q + 1], m * acc[a][4 * q + 2],
                                    m * acc[a][4 * q + 3]);
                }
            }
        }
        if (norm) {  // z is read by the normalised map only
            if (tid < D) {
                const float lend = LT[tid * LDT + n - 1];
                const float gz = expf(lend);
                float zz = split ? sz[tid] : gz * sz[tid];
                for (int j = 0; j < kSub; ++j)
                    zz += split ? kT[tid * LDT + j]
                                : kT[tid * LDT + j] * __expf(lend - LT[tid * LDT + j]);
                sz[tid] = split ? gz * zz : zz;
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
    const size_t st_smem = sizeof(float) * ((size_t)kSub * (2 * D + DV + 8) + 2 * D);
    cudaError_t err = cudaFuncSetAttribute(k_gla_state<D, DV, T>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st_smem);
    if (err != cudaSuccess)
        return err;
    k_gla_state<D, DV, T><<<(unsigned)(BH * nblk), kThreads, st_smem, a.stream>>>(
        k, v, a.alpha, ws, dec, a.N, nblk, a.fm);
    count_launches(1);
    err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    const int per_seq = (E + kThreads - 1) / kThreads;
    k_gla_scan<<<(unsigned)(BH * per_seq), kThreads, 0, a.stream>>>(ws, dec, nblk, D, DV);
    count_launches(1);
    err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    constexpr int NH = DV > 64 ? DV / 64 : 1;
    const size_t smem = GlaOut<D, DV / NH>::bytes;
    auto kern = k_gla_out<D, DV, T>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess)
        return err;
    kern<<<(unsigned)(BH * nblk * NH), kThreads, smem, a.stream>>>(q, k, v, a.alpha, a.out, ws, a.N,
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
