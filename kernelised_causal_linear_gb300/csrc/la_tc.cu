// la_tc.cu -- single-pass causal forward on the tcgen05 tensor cores
// (bf16 q/k/v, d = dv = 64, no decay).
//
// The sequence is cut into chunks of C = 128 tokens ("Efficient Attention
// Variants", section 8: parallel inside a chunk, state passed between chunks;
// "Linear Attention and SSM", eq. attn-linssm-ssd: inside a chunk the output
// is the masked form ((phi(Q) phi(K)^T) o L) V with L the causal mask).  For a
// chunk with queries Q_c, keys K_c, values V_c and the state S_prev, z_prev of
// every earlier token:
//
//   P     = tril(phi(Q_c) phi(K_c)^T)                      (fp32, tensor memory)
//   num   = P V_c + phi(Q_c) S_prev                        (tensor cores)
//   den   = rowsum(P) + phi(Q_c) z_prev                    (CUDA cores, fp32)
//   o     = num / max(den, FLT_MIN)
//   dS_c  = phi(K_c)^T V_c,  dz_c = column sums of phi(K_c)
//
// ("Linear Attention Kernel", section "Rewrite: associativity": phi(K)^T V
// is the only intermediate; "Efficient Attention Variants", section 5: the
// prefix state S_t, z_t and the normalised read).
//
// Chunks are grouped into segments of L consecutive chunks of one sequence.
// One persistent CTA per SM takes segments in ticket order (segment-major over
// the B*H sequences) and runs each in two phases:
//   A  the segment's aggregate: K, V of every chunk (kept in L2 with an
//      evict-last hint), phi(K), dS accumulated on the tensor cores, dz;
//      published at once to a ring of per-segment slots in global memory;
//   C  the outputs: Q, K, V again (K, V from L2), with the running state
//      S_prev = S_in + the segment's earlier chunks carried in tensor memory.
// Between them a decoupled look-back over the predecessors' slots gives S_in,
// the state before the segment, and publishes the segment's inclusive prefix.
// Phase A of segment j+1 runs before phase C of segment j, so the look-back
// of segment j is hidden behind it.  The look-back starts from the nearest
// inclusive prefix and adds later aggregates in segment order, so every
// prefix is the same left-to-right fp32 sum whatever the timing: results are
// bitwise reproducible.
//
// The CTA is warp-specialised; work flows through rings of shared-memory
// stages and tensor-memory buffers, synchronised by mbarriers:
//   warp 0      producer: segment tickets, TMA loads
//   warp 1      MMA issuer: segment aggregate, scores, chunk state, P V,
//               phi(Q) S_prev
//   warps 2-3   look-back over the predecessors' slots, S_in, inclusive prefix
//   warps 4-7   phi(K) in place and its column sums (phases A and C); P:
//               causal mask, row sums, bf16 hi/lo re-pack in tensor memory
//   warps 8-11  segment aggregate out of tensor memory and published; running
//               state S_prev as bf16 hi/lo for the tensor cores, z_prev
//   warps 12-15 phi(Q) in place (one chunk ahead), epilogue: denominator,
//               output tile by TMA store
//
// Precision: phi(Q), phi(K) and V enter the MMAs as bf16 (phi rounded once);
// P and S_prev are fp32 and enter as a bf16 hi/lo pair (two MMAs each), so
// their rounding is ~2^-17 relative; states and denominators stay fp32.
//
// Operands: Q, K, V chunks arrive by TMA in the 128-byte swizzled layout.
// The scores MMA reads Q and K K-major; the state MMAs read [V | phi(K)] as an
// MN-major A of 128 rows (the second 64 rows are discarded) against phi(K)
// MN-major, giving dS^T in lanes 0..63; P's hi/lo parts sit in tensor memory
// as the A operand of P V; S_prev^T hi/lo sit in shared memory K-major for
// phi(Q) S_prev.
//
// Every wait is bounded (%globaltimer); on expiry the CTA records
// LA_ERR_TIMEOUT, every role leaves its loop, the CTA drains its own TMA loads,
// MMAs and stores, frees its tensor memory and exits.
#include <cudaTypedefs.h>
#include <algorithm>
#include <float.h>
#include <mutex>
#include <string.h>

#include "la_internal.cuh"
#include "la_sm100.cuh"

namespace la {
namespace {

using namespace sm100;

constexpr int kC = 128;        // tokens per chunk
constexpr int kD = 64;         // d = dv
constexpr int kThreads = 512;  // 16 warps
constexpr int NQ = 3;          // Q stages
constexpr int NKV = 3;         // K,V stages
constexpr int NS = 4;          // segment-ticket ring
constexpr int kStateFloats = kD * kD + kD;         // S^T (dv x d) then z (d)
constexpr int kSlotFloats = 2 * kStateFloats;      // aggregate, inclusive
constexpr int kMaxList = 128;                      // look-back entries
constexpr uint64_t kWaitNs = 2000000000ull;        // 2 s for any single wait

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;                          // NQ x (128 x 64 bf16)
constexpr uint32_t OFF_KV = OFF_Q + NQ * 16384;        // NKV x (V then K)
constexpr uint32_t OFF_S = OFF_KV + NKV * 32768;       // 2 x (S^T hi, S^T lo)
constexpr uint32_t OFF_O = OFF_S + 2 * 16384;          // output staging 2 x 16 KiB
constexpr uint32_t OFF_MISC = OFF_O + 32768;
constexpr uint32_t kMiscBytes = 16384;
constexpr int kMaxL = 8;       // largest segment (chunks)
constexpr int NPH = 4;         // phi(K) scratch ring depth, in segments
constexpr uint32_t SMEM_BYTES = OFF_MISC + kMiscBytes + 1024;  // + alignment slack

// tensor memory columns
constexpr uint32_t TM_P = 0;       // scores fp32, 128 columns
constexpr uint32_t TM_PHL = 128;   // P hi (128..191), P lo (192..255), bf16 pairs
constexpr uint32_t TM_O = 256;     // 2 x 64: output accumulators
constexpr uint32_t TM_SRUN = 384;  // running S_prev^T (lanes 0..63)
constexpr uint32_t TM_DSEG = 448;  // segment aggregate dS^T (lanes 0..63)

struct TcParams {
    CUtensorMap mq, mk, mv, mo;
    CUtensorMap mphi;  // phi(K) scratch: per CTA NPH x L tiles of 128 x 64 bf16
    int64_t N;
    int BH;
    int nchunk;   // chunks per sequence
    int L;        // chunks per segment
    int nseg;     // segments per sequence
    int R;        // ring slots per sequence
    int total;    // BH * nseg segment tickets
    int fm;
    unsigned* counter;
    unsigned* flags;
    float* slots;
    float* sin_scratch;  // per CTA: 2 x S_in
    void* phi_scratch;   // the tiles mphi describes
    int* status;
};

struct Misc {
    uint64_t seg_full[NS], seg_empty[NS];
    uint64_t q_full[NQ], q_empty[NQ], q_phi[NQ];
    uint64_t kv_full[NKV], kv_empty[NKV], aphi[NKV], phik_stored[NPH];
    uint64_t mma1_done[2], p_ready[2], pv_done[2], srun_read[2], o_done[2], o_free[2];
    uint64_t epi_done[2];
    uint64_t dseg_done, dseg_free, dzseg_ready[2], agg_pub[2], sin_ready[2], sin_free[2];
    uint64_t drain;
    uint32_t tmem;
    int abort;
    int seg_ticket[NS];
    int nlist;
    int list[kMaxList];
    float den[2][kC];
    alignas(16) float zprev[2][kD];
    float zrun[kD];
    float dza[4][kD];        // per A chunk: column sums of phi(K), one row per warp
    float dzacc[kD];         // running column sums over the current A segment
    float dzk[NPH][kMaxL][kD];  // per chunk column sums, kept for phase C
    float dzseg[2][kD];
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc");

// Optional per-chunk event timestamps (SM clock) for pipeline analysis; only
// in builds with LA_TC_TRACE defined, never in the library as shipped.
#ifdef LA_TC_TRACE
__device__ unsigned long long* g_tc_trace;
#define TC_TRACE(i, ev)                                                                       \
    do {                                                                                      \
        if (g_tc_trace && (i) < 64)                                                           \
            g_tc_trace[(static_cast<size_t>(blockIdx.x) * 64 + (i)) * 16 + (ev)] = clock64(); \
    } while (0)
#else
#define TC_TRACE(i, ev) \
    do {                \
    } while (0)
#endif

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void named_bar(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    uint64_t t0 = 0;
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_sleep(bar, parity, 20000u))
            return true;
        if ((n & 3u) == 0u) {
            if (*abort)
                return false;
            const uint64_t now = globaltimer();
            if (!t0)
                t0 = now;
            else if (now - t0 > kWaitNs) {
                *abort = 1;
                return false;
            }
        }
    }
}

// A thread group waits through one leader; bar.red hands every thread the
// same verdict, so the group never splits on an abort.
__device__ __forceinline__ bool group_ok(int ok, int barid, int count)
{
    int res;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, p;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(res)
        : "r"(ok), "r"(barid), "r"(count)
        : "memory");
    return res != 0;
}

// Bounded wait used only while draining (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kWaitNs)
            return;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t bf2_min0(uint32_t w)
{
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0u));
    return r;
}

__device__ __forceinline__ uint32_t bf2_max0(uint32_t w)
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0u));
    return r;
}

__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// elu(x)+1 on two packed bf16: max(x,0) + exp(min(x,0)).  One of the two
// terms is always exact (0, or exp(0) = 1), so rounding exp(min(x,0)) to bf16
// first and adding in bf16 gives the correctly rounded result of the fp32 sum.
__device__ __forceinline__ uint32_t phi2(uint32_t w)
{
    const uint32_t mn = bf2_min0(w);
    return bf2_add(bf2_max0(w), pack_bf16x2(__expf(bf_lo(mn)), __expf(bf_hi(mn))));
}

// split two fp32 into packed bf16 hi and lo parts
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo)
{
    hi = pack_bf16x2(a, b);
    lo = pack_bf16x2(a - bf_lo(hi), b - bf_hi(hi));
}

// Feature map in place on a 128 x 64 bf16 tile (128-byte swizzle) by 128
// threads; rows >= valid become zero.  With zsum, also the column sums of the
// result: zsum[warp][64] (rows of this warp's threads only).  With gdst, the
// result is also written to global memory as a plain row-major 128 x 64 tile.
__device__ __noinline__ void phi_tile(unsigned char* tile, int t, int valid, bool elu,
                                     float (*zsum)[kD], uint4* gdst)
{
    const int cc = t & 7, r0 = t >> 3;
    uint4 x[8];
#pragma unroll
    for (int mm = 0; mm < 8; ++mm)
        x[mm] = *reinterpret_cast<const uint4*>(tile + sw128_off(r0 + 16 * mm, cc));
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) {
        const int r = r0 + 16 * mm;
        if (r >= valid)
            x[mm] = make_uint4(0, 0, 0, 0);
        else if (elu)
            x[mm] = make_uint4(phi2(x[mm].x), phi2(x[mm].y), phi2(x[mm].z), phi2(x[mm].w));
        if (r >= valid || elu)
            *reinterpret_cast<uint4*>(tile + sw128_off(r, cc)) = x[mm];
        if (gdst)
            gdst[r * 8 + cc] = x[mm];
    }
    if (zsum) {
        float zp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            zp[e] = 0.f;
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
            zp[0] += bf_lo(x[mm].x), zp[1] += bf_hi(x[mm].x);
            zp[2] += bf_lo(x[mm].y), zp[3] += bf_hi(x[mm].y);
            zp[4] += bf_lo(x[mm].z), zp[5] += bf_hi(x[mm].z);
            zp[6] += bf_lo(x[mm].w), zp[7] += bf_hi(x[mm].w);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            zp[e] += __shfl_xor_sync(0xffffffffu, zp[e], 8);
            zp[e] += __shfl_xor_sync(0xffffffffu, zp[e], 16);
        }
        if ((t & 31) < 8)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                zsum[(t >> 5) & 3][8 * cc + e] = zp[e];
    }
}

// Segment helpers
struct Seg {
    int t;       // ticket
    int s;       // sequence
    int c0;      // first chunk
    int n;       // chunks in this segment
};

__device__ __forceinline__ Seg seg_of(const TcParams& p, int t)
{
    Seg g;
    g.t = t;
    const int gi = t / p.BH;
    g.s = t % p.BH;
    g.c0 = gi * p.L;
    g.n = min(p.L, p.nchunk - g.c0);
    return g;
}

__device__ __forceinline__ int chunk_valid(const TcParams& p, int c)
{
    return static_cast<int>(min(static_cast<int64_t>(kC), p.N - static_cast<int64_t>(c) * kC));
}

// Job order shared by every role.  Round j holds phase A of local segment j
// and phase C of local segment j-2, interleaved chunk by chunk
// (A0 C0 A1 C1 ...); the two rounds between a segment's phases hide its
// look-back.
struct Round {
    int j;        // round = local index of the A segment
    int tA, tC;   // tickets of the A and C segments (-1: none)
    Seg gA, gC;
    int nA, nC;
};

__device__ __forceinline__ void round_setup(const TcParams& p, Round& r, int j, int tA, int tC)
{
    r.j = j;
    r.tA = tA;
    r.tC = tC;
    r.nA = r.nC = 0;
    if (tA >= 0) {
        r.gA = seg_of(p, tA);
        r.nA = r.gA.n;
    }
    if (tC >= 0) {
        r.gC = seg_of(p, tC);
        r.nC = r.gC.n;
    }
}

__global__ void __launch_bounds__(kThreads, 1) k_fwd_tc64(const __grid_constant__ TcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Misc* m = reinterpret_cast<Misc*>(sm + OFF_MISC);
    volatile int* abort = &m->abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool norm = p.fm != LA_FM_NONE;
    const bool elu = p.fm == LA_FM_ELU1;

    if (tid == 0) {
        uint64_t* bars = reinterpret_cast<uint64_t*>(m);
        const int nbars = static_cast<int>((reinterpret_cast<uint64_t*>(&m->drain) - bars) + 1);
        for (int i = 0; i < nbars; ++i)
            mbar_init(&bars[i], 1);
        m->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.mq);
        tma_prefetch_desc(&p.mk);
        tma_prefetch_desc(&p.mv);
        tma_prefetch_desc(&p.mo);
        tma_prefetch_desc(&p.mphi);
    }
    if (tid < kD)
        m->dzacc[tid] = 0.f;
    if (warp == 0) {
        tmem_alloc(&m->tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = m->tmem;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // phi(K) scratch tile of local segment jj, chunk k
    auto phi_index = [&](int jj, int k) {
        return (static_cast<int>(blockIdx.x) * NPH + jj % NPH) * p.L + k;
    };

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            const uint64_t keep = policy_evict_last();
            const uint64_t stream = policy_evict_first();
            int q_last[NQ], kv_last[NKV];
            for (int j = 0; j < NQ; ++j)
                q_last[j] = -1;
            for (int j = 0; j < NKV; ++j)
                kv_last[j] = -1;
            int kvi = 0, ci = 0, h1 = -1, h2 = -1;
            bool ok = true, doneA = false;
            // K (or, in phase C, phi(K) from the scratch tile `phi`) and V
            auto load_kv = [&](const Seg& g, int c, uint64_t pol, int phi) -> bool {
                const int ks = kvi % NKV;
                if (kvi >= NKV && !bwait(&m->kv_empty[ks], ((kvi / NKV) & 1) ^ 1, abort))
                    return false;
                mbar_arrive_expect_tx(&m->kv_full[ks], 2 * kC * kD * 2);
                unsigned char* kv = sm + OFF_KV + ks * 32768;
                if (phi >= 0)
                    tma_load_3d(kv + 16384, &p.mphi, 0, 0, phi, &m->kv_full[ks], pol);
                else
                    tma_load_3d(kv + 16384, &p.mk, 0, c * kC, g.s, &m->kv_full[ks], pol);
                tma_load_3d(kv, &p.mv, 0, c * kC, g.s, &m->kv_full[ks], pol);
                kv_last[ks] = kvi / NKV;
                ++kvi;
                return true;
            };
            for (int j = 0; ok; ++j) {
                int tA = -1;
                if (!doneA) {
                    const int t = static_cast<int>(atomicAdd(p.counter, 1u));
                    const int ss = j % NS;
                    if (j >= NS && !bwait(&m->seg_empty[ss], ((j / NS) & 1) ^ 1, abort))
                        break;
                    m->seg_ticket[ss] = t;
                    mbar_arrive(&m->seg_full[ss]);
                    if (t < p.total)
                        tA = t;
                    else
                        doneA = true;
                }
                Round r;
                round_setup(p, r, j, tA, h2);
                if (r.nA == 0 && r.nC == 0 && h1 < 0)
                    break;
                const int jc = j - 2;
                if (r.nC && !bwait(&m->phik_stored[jc % NPH], (jc / NPH) & 1, abort))
                    break;
                for (int k = 0; k < max(r.nA, r.nC) && ok; ++k) {
                    if (k < r.nA)
                        ok = load_kv(r.gA, r.gA.c0 + k, keep, -1);
                    if (k < r.nC && ok) {
                        const int qs = ci % NQ;
                        if (ci >= NQ && !bwait(&m->q_empty[qs], ((ci / NQ) & 1) ^ 1, abort)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&m->q_full[qs], kC * kD * 2);
                        tma_load_3d(sm + OFF_Q + qs * 16384, &p.mq, 0, (r.gC.c0 + k) * kC,
                                    r.gC.s, &m->q_full[qs], stream);
                        q_last[qs] = ci / NQ;
                        TC_TRACE(ci, 0);
                        ++ci;
                        ok = load_kv(r.gC, r.gC.c0 + k, stream, phi_index(jc, k));
                    }
                }
                h2 = h1;
                h1 = tA;
            }
            if (*abort) {  // let every load this thread issued land before exit
                for (int j = 0; j < NQ; ++j)
                    if (q_last[j] >= 0)
                        drain_wait(&m->q_full[j], q_last[j] & 1);
                for (int j = 0; j < NKV; ++j)
                    if (kv_last[j] >= 0)
                        drain_wait(&m->kv_full[j], kv_last[j] & 1);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer --
        if (lane == 0) {
            const uint32_t id_sc = idesc_bf16_f32(128, 128, false, false);
            const uint32_t id_st = idesc_bf16_f32(128, 64, true, true);
            const uint32_t id_pv = idesc_bf16_f32(128, 64, false, true);
            const uint32_t id_in = idesc_bf16_f32(128, 64, false, false);
            // Operand descriptors of stage 0; a stage or K-step offset of x bytes
            // adds x >> 4 to the start-address field.
            const uint64_t dq0 = sdesc_sw128(smem_addr(sm + OFF_Q), 16, 1024);
            const uint32_t v0 = smem_addr(sm + OFF_KV);
            const uint64_t dk0 = sdesc_sw128(v0 + 16384, 16, 1024);
            const uint64_t dvm0 = sdesc_sw128(v0, 16384, 1024);  // [V | phi(K)]: one 128-row A
            const uint64_t dvb0 = sdesc_sw128(v0, 16, 1024);
            const uint64_t ds0 = sdesc_sw128(smem_addr(sm + OFF_S), 16, 1024);
            auto dq = [&](int i) { return dq0 + (uint64_t)(i * (16384 >> 4)); };
            auto dk = [&](int i) { return dk0 + (uint64_t)(i * (32768 >> 4)); };
            auto dvm = [&](int i) { return dvm0 + (uint64_t)(i * (32768 >> 4)); };
            auto dvb = [&](int i) { return dvb0 + (uint64_t)(i * (32768 >> 4)); };
            auto ds = [&](int i) { return ds0 + (uint64_t)(i * (16384 >> 4)); };
            bool issued = false, ok = true, doneA = false;
            int kvi = 0, ci = 0, ai = 0, nsegA = 0, h1 = -1, h2 = -1;
            // [V | phi(K)]^T phi(K) of stage ks accumulated into d
            auto state_mma = [&](uint32_t d, int ks, bool acc) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ss(d, dvm(ks) + 128 * kk, dk(ks) + 128 * kk, id_st, acc || kk > 0);
            };
            for (int j = 0; ok; ++j) {
                int tA = -1;
                if (!doneA) {
                    if (!bwait(&m->seg_full[j % NS], (j / NS) & 1, abort))
                        break;
                    const int t = m->seg_ticket[j % NS];
                    if (t < p.total)
                        tA = t;
                    else
                        doneA = true;
                }
                Round r;
                round_setup(p, r, j, tA, h2);
                if (r.nA == 0 && r.nC == 0 && h1 < 0)
                    break;
                for (int k = 0; k < max(r.nA, r.nC) && ok; ++k) {
                    if (k < r.nA) {  // phase A: segment aggregate into TM_DSEG
                        const int ks = kvi % NKV;
                        if ((k == 0 && nsegA >= 1 &&
                             !bwait(&m->dseg_free, (nsegA - 1) & 1, abort)) ||
                            !bwait(&m->aphi[ai % NKV], (ai / NKV) & 1, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        state_mma(tm + TM_DSEG, ks, k > 0);
                        mma_commit(&m->kv_empty[ks]);
                        issued = true;
                        ++kvi, ++ai;
                        if (k == r.nA - 1) {
                            mma_commit(&m->dseg_done);
                            ++nsegA;
                        }
                    }
                    if (k < r.nC) {  // phase C: one chunk of outputs
                        const int b = ci & 1, qs = ci % NQ, ks = kvi % NKV;
                        if (!bwait(&m->q_phi[qs], (ci / NQ) & 1, abort) ||
                            !bwait(&m->kv_full[ks], (kvi / NKV) & 1, abort) ||
                            !bwait(&m->srun_read[b], (ci >> 1) & 1, abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ss(tm + TM_P, dq(qs) + 2 * kk, dk(ks) + 2 * kk, id_sc, kk > 0);
                        state_mma(tm + TM_SRUN, ks, true);
                        mma_commit(&m->mma1_done[b]);
                        TC_TRACE(ci, 7);
                        issued = true;
                        if (!bwait(&m->p_ready[b], (ci >> 1) & 1, abort) ||
                            (ci >= 2 && !bwait(&m->o_free[b], ((ci >> 1) & 1) ^ 1, abort))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        TC_TRACE(ci, 14);
                        const uint32_t o = tm + TM_O + 64 * b;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16_ts(o, tm + TM_PHL + 8 * kk, dvb(ks) + 128 * kk, id_pv, kk > 0);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16_ts(o, tm + TM_PHL + 64 + 8 * kk, dvb(ks) + 128 * kk, id_pv, 1);
                        mma_commit(&m->pv_done[b]);
                        mma_commit(&m->kv_empty[ks]);
                        TC_TRACE(ci, 8);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ss(o, dq(qs) + 2 * kk, ds(b) + 2 * kk, id_in, 1);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ss(o, dq(qs) + 2 * kk, ds(b) + 512 + 2 * kk, id_in, 1);
                        mma_commit(&m->o_done[b]);
                        TC_TRACE(ci, 9);
                        ++ci, ++kvi;
                    }
                }
                h2 = h1;
                h1 = tA;
            }
            if (issued && *abort) {  // every MMA issued here retires before tensor memory is freed
                mma_commit(&m->drain);
                drain_wait(&m->drain, 0);
            }
        }
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------ look-back, S_in (warps 2-3) --
        const int tl = tid - 64;  // 0..63
        const bool lead = tl == 0;
        const unsigned full = 0xffffffffu;
        for (int j = 0;; ++j) {
            const int ss = j % NS;
            if (!group_ok(!lead || bwait(&m->seg_full[ss], (j / NS) & 1, abort), 4, 64))
                break;
            const int t = m->seg_ticket[ss];
            if (t >= p.total)
                break;
            const Seg g = seg_of(p, t);
            const int gi = t / p.BH;
            if (!group_ok(!lead || j < 2 || bwait(&m->sin_free[j & 1], ((j >> 1) & 1) ^ 1, abort),
                          4, 64))
                break;
            const unsigned* flag_base = p.flags + static_cast<size_t>(g.s) * p.R;
            float* slot_base = p.slots + static_cast<size_t>(g.s) * p.R * kSlotFloats;
            if (warp == 2) {
                // Lane l watches segment base - l.  With a wrapping ring only R-1
                // slots behind this segment are distinct from its own; a slot
                // holding another epoch reads as not ready.
                const int W = p.R >= p.nseg ? 32 : min(32, p.R - 1);
                const unsigned active = W >= 32 ? 0xffffffffu : ((1u << W) - 1u);
                int n = 0, base = gi - 1;
                uint64_t start = 0;
                while (base >= 0) {
                    const int pg = base - lane;
                    bool ready = true, incl = true;
                    if (lane >= W) {
                        ready = incl = false;
                    } else if (pg >= 0) {
                        const unsigned f = ld_acquire(flag_base + pg % p.R);
                        ready = (f >> 2) == static_cast<unsigned>(pg + 1) && (f & 3u) != 0u;
                        incl = ready && (f & 3u) == 2u;
                    }
                    const unsigned mi = __ballot_sync(full, incl) & active;
                    const unsigned mr = __ballot_sync(full, ready) & active;
                    if (mi) {
                        const int ls = __ffs(mi) - 1;
                        const unsigned need = ls == 0 ? 0u : ((1u << ls) - 1u);
                        if ((mr & need) == need) {
                            if (n + ls + 1 > kMaxList) {
                                n = -2;
                                break;
                            }
                            if (lane < ls)
                                m->list[n + lane] = (pg % p.R) << 1;
                            if (lane == ls && pg >= 0)
                                m->list[n + lane] = ((pg % p.R) << 1) | 1;
                            n += ls + (base - ls >= 0 ? 1 : 0);
                            break;
                        }
                    } else if (mr == active) {
                        if (n + W > kMaxList) {
                            n = -2;
                            break;
                        }
                        if (lane < W)
                            m->list[n + lane] = (pg % p.R) << 1;
                        n += W;
                        base -= W;
                        start = 0;
                        continue;
                    }
                    const uint64_t now = globaltimer();
                    if (!start)
                        start = now;
                    if (__any_sync(full, now - start > kWaitNs || *abort)) {
                        n = -1;
                        break;
                    }
                    __nanosleep(200);
                }
                if (lane == 0) {
                    m->nlist = n;
                    if (n < 0) {
                        set_status(p.status, n == -1 ? LA_ERR_TIMEOUT : LA_ERR_DEVICE_CHECK);
                        *abort = 1;
                    }
                }
            }
            named_bar(4, 64);
            const int nlist = m->nlist;
            if (nlist < 0)
                break;
            // S_in: the nearest inclusive prefix plus the later aggregates in
            // segment order; thread tl owns float4 words tl + 64 u, u = 0..16.
            float4 acc[17];
#pragma unroll
            for (int u = 0; u < 17; ++u)
                acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int e = nlist - 1; e >= 0; --e) {
                const int ent = m->list[e];
                const float4* src = reinterpret_cast<const float4*>(
                    slot_base + static_cast<size_t>(ent >> 1) * kSlotFloats +
                    ((ent & 1) ? kStateFloats : 0));
#pragma unroll
                for (int u = 0; u < 17; ++u) {
                    const int f = tl + 64 * u;
                    if (f < kStateFloats / 4) {
                        const float4 x = __ldcg(src + f);
                        acc[u].x += x.x, acc[u].y += x.y, acc[u].z += x.z, acc[u].w += x.w;
                    }
                }
            }
            float4* sin = reinterpret_cast<float4*>(
                p.sin_scratch + (static_cast<size_t>(blockIdx.x) * 2 + (j & 1)) * kStateFloats);
#pragma unroll
            for (int u = 0; u < 17; ++u) {
                const int f = tl + 64 * u;
                if (f < kStateFloats / 4)
                    __stcg(sin + f, acc[u]);
            }
            // the inclusive prefix needs this segment's own aggregate
            if (!group_ok(!lead || bwait(&m->agg_pub[j & 1], (j >> 1) & 1, abort), 4, 64))
                break;
            const int my = gi % p.R;
            const float4* agg =
                reinterpret_cast<const float4*>(slot_base + static_cast<size_t>(my) * kSlotFloats);
            float4* inc = reinterpret_cast<float4*>(slot_base + static_cast<size_t>(my) * kSlotFloats +
                                                    kStateFloats);
#pragma unroll
            for (int u = 0; u < 17; ++u) {
                const int f = tl + 64 * u;
                if (f < kStateFloats / 4) {
                    const float4 a = __ldcg(agg + f);
                    __stcg(inc + f, make_float4(acc[u].x + a.x, acc[u].y + a.y, acc[u].z + a.z,
                                                acc[u].w + a.w));
                }
            }
            named_bar(4, 64);
            if (lead) {
                __threadfence();
                st_release(const_cast<unsigned*>(flag_base) + my,
                           (static_cast<unsigned>(gi + 1) << 2) | 2u);
                mbar_arrive(&m->sin_ready[j & 1]);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------------------------- P, epilogue (warps 4-7) --------
        const int ta = tid - 128;
        const bool lead = ta == 0;
        const uint64_t pol = policy_evict_first();
        unsigned char* sO = sm + OFF_O;
        int ci = 0, h1 = -1, h2 = -1;
        bool doneA = false;
        // the epilogue of a chunk runs after P of the next one; its row sum of P
        // (the intra-chunk denominator) waits in a register
        int pend_ci = -1, pend_c = 0, pend_s = 0, pend_last = 0, pend_ss = 0;
        float pend_rs = 0.f;
        auto epilogue = [&]() -> bool {
            const int cj = pend_ci, b = cj & 1, qs = cj % NQ;
            if (!group_ok(!lead || (bwait(&m->q_phi[qs], (cj / NQ) & 1, abort) &&
                                    bwait(&m->srun_read[b], (cj >> 1) & 1, abort) &&
                                    bwait(&m->o_done[b], (cj >> 1) & 1, abort)),
                          1, 128))
                return false;
            tc_fence_after();
            if (lead)
                TC_TRACE(cj, 5);
            float den = pend_rs;
            if (norm) {
                const unsigned char* sQ = sm + OFF_Q + qs * 16384;
                const float* z = m->zprev[b];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 x = *reinterpret_cast<const uint4*>(sQ + sw128_off(ta, cc));
                    const float4 z0 = *reinterpret_cast<const float4*>(z + 8 * cc);
                    const float4 z1 = *reinterpret_cast<const float4*>(z + 8 * cc + 4);
                    den = fmaf(bf_lo(x.x), z0.x, den);
                    den = fmaf(bf_hi(x.x), z0.y, den);
                    den = fmaf(bf_lo(x.y), z0.z, den);
                    den = fmaf(bf_hi(x.y), z0.w, den);
                    den = fmaf(bf_lo(x.z), z1.x, den);
                    den = fmaf(bf_hi(x.z), z1.y, den);
                    den = fmaf(bf_lo(x.w), z1.z, den);
                    den = fmaf(bf_hi(x.w), z1.w, den);
                }
            }
            const float inv = norm ? 1.0f / fmaxf(den, FLT_MIN) : 1.0f;
            if (lead)
                bulk_wait_read<0>();  // the previous tile has left the staging buffer
            named_bar(1, 128);
            uint32_t rr[4][16];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tmem_ld16(tm + TM_O + 64 * b + lane_off + 16 * q, rr[q]);
            tmem_ld_wait();
            if (lead)
                TC_TRACE(cj, 13);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int col4 = 4 * q + u;
                    const float4 o = make_float4(__uint_as_float(rr[q][4 * u]) * inv,
                                                 __uint_as_float(rr[q][4 * u + 1]) * inv,
                                                 __uint_as_float(rr[q][4 * u + 2]) * inv,
                                                 __uint_as_float(rr[q][4 * u + 3]) * inv);
                    *reinterpret_cast<float4*>(sO + (col4 >> 3) * 16384 +
                                               sw128_off(ta, col4 & 7)) = o;
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar(1, 128);
            if (lead) {
                mbar_arrive(&m->o_free[b]);
                mbar_arrive(&m->q_empty[qs]);
                mbar_arrive(&m->epi_done[b]);
                if (pend_last)
                    mbar_arrive(&m->seg_empty[pend_ss]);
                tma_store_3d(&p.mo, sO, 0, pend_c * kC, pend_s, pol);
                tma_store_3d(&p.mo, sO + 16384, 32, pend_c * kC, pend_s, pol);
                bulk_commit();
                TC_TRACE(cj, 15);
            }
            pend_ci = -1;
            return true;
        };
        bool ok = true;
        for (int j = 0; ok; ++j) {
            int tA = -1;
            if (!doneA) {
                if (!group_ok(!lead || bwait(&m->seg_full[j % NS], (j / NS) & 1, abort), 1, 128))
                    break;
                const int t = m->seg_ticket[j % NS];
                if (t < p.total)
                    tA = t;
                else
                    doneA = true;
            }
            Round r;
            round_setup(p, r, j, tA, h2);
            if (r.nA == 0 && r.nC == 0 && h1 < 0)
                break;
            for (int k = 0; k < r.nC; ++k, ++ci) {
                const int b = ci & 1;
                // P: causal mask, row sums, bf16 hi/lo into TM_PHL
                if (!group_ok(!lead || (bwait(&m->mma1_done[b], (ci >> 1) & 1, abort) &&
                                        (ci < 1 || bwait(&m->pv_done[(ci - 1) & 1],
                                                         ((ci - 1) >> 1) & 1, abort))),
                              1, 128)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lead)
                    TC_TRACE(ci, 3);
                float rs = 0.f;
                // rows 0..63 see only keys 0..63: the upper 64 columns are masked
                const int nq = ta < 64 ? 2 : 4;
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t hi[16], lo[16];
                    if (q < nq) {
                        uint32_t v0[16], v1[16];
                        tmem_ld16(tm + TM_P + lane_off + 32 * q, v0);
                        tmem_ld16(tm + TM_P + lane_off + 32 * q + 16, v1);
                        tmem_ld_wait();
                        const int lim = ta - 32 * q;  // keys jj <= ta stay
#pragma unroll
                        for (int mm = 0; mm < 8; ++mm) {
                            const float a = 2 * mm <= lim ? __uint_as_float(v0[2 * mm]) : 0.f;
                            const float bb =
                                2 * mm + 1 <= lim ? __uint_as_float(v0[2 * mm + 1]) : 0.f;
                            rs += a + bb;
                            split2(a, bb, hi[mm], lo[mm]);
                        }
#pragma unroll
                        for (int mm = 0; mm < 8; ++mm) {
                            const float a =
                                16 + 2 * mm <= lim ? __uint_as_float(v1[2 * mm]) : 0.f;
                            const float bb =
                                17 + 2 * mm <= lim ? __uint_as_float(v1[2 * mm + 1]) : 0.f;
                            rs += a + bb;
                            split2(a, bb, hi[8 + mm], lo[8 + mm]);
                        }
                    } else {
#pragma unroll
                        for (int mm = 0; mm < 16; ++mm)
                            hi[mm] = lo[mm] = 0u;
                    }
                    tmem_st16(tm + TM_PHL + lane_off + 16 * q, hi);
                    tmem_st16(tm + TM_PHL + lane_off + 64 + 16 * q, lo);
                }
                tmem_st_wait();
                if (lead)
                    TC_TRACE(ci, 10);
                tc_fence_before();
                named_bar(1, 128);
                if (lead) {
                    mbar_arrive(&m->p_ready[b]);
                    TC_TRACE(ci, 6);
                }
                if (pend_ci >= 0 && !epilogue()) {
                    ok = false;
                    break;
                }
                pend_ci = ci, pend_c = r.gC.c0 + k, pend_s = r.gC.s, pend_rs = rs;
                pend_last = k == r.nC - 1, pend_ss = (j - 2) % NS;
            }
            h2 = h1;
            h1 = tA;
        }
        if (ok && pend_ci >= 0)
            epilogue();
        if (lead)
            bulk_wait<0>();
    } else if (warp >= 8 && warp < 12) {
        // ------------- phi(K), segment aggregate, S_prev (warps 8-11) ------
        const int tb = tid - 256, wb = warp - 8;
        const bool lead = tb == 0;
        int kvi = 0, ci = 0, ai = 0, nsegA = 0, h1 = -1, h2 = -1;
        bool ok = true, doneA = false;
        for (int j = 0; ok; ++j) {
            int tA = -1;
            if (!doneA) {
                if (!group_ok(!lead || bwait(&m->seg_full[j % NS], (j / NS) & 1, abort), 2, 128))
                    break;
                const int t = m->seg_ticket[j % NS];
                if (t < p.total)
                    tA = t;
                else
                    doneA = true;
            }
            Round r;
            round_setup(p, r, j, tA, h2);
            if (r.nA == 0 && r.nC == 0 && h1 < 0)
                break;
            const int jc = j - 2;
            for (int k = 0; k < max(r.nA, r.nC) && ok; ++k) {
                if (k < r.nA) {  // phase A: phi(K) kept for phase C, column sums
                    const int ks = kvi % NKV;
                    if (!group_ok(!lead || bwait(&m->kv_full[ks], (kvi / NKV) & 1, abort), 2,
                                  128)) {
                        ok = false;
                        break;
                    }
                    unsigned char* ktile = sm + OFF_KV + ks * 32768 + 16384;
                    if (lead)
                        TC_TRACE(ai, 2);
                    // phi(K) is kept for phase C in the scratch (plain stores,
                    // fenced before the TMA loads of phase C read it)
                    phi_tile(ktile, tb, chunk_valid(p, r.gA.c0 + k), elu, m->dza,
                             reinterpret_cast<uint4*>(p.phi_scratch) +
                                 static_cast<size_t>(phi_index(j, k)) * (kC * kD * 2 / 16));
                    fence_proxy_async_smem();
                    named_bar(2, 128);
                    if (tb < kD) {
                        const float dz =
                            m->dza[0][tb] + m->dza[1][tb] + m->dza[2][tb] + m->dza[3][tb];
                        m->dzacc[tb] += dz;
                        m->dzk[j % NPH][k][tb] = dz;
                    }
                    if (lead) {
                        mbar_arrive(&m->aphi[ai % NKV]);
                        TC_TRACE(ai, 11);
                    }
                    named_bar(2, 128);
                    ++kvi, ++ai;
                    if (k == r.nA - 1) {  // segment aggregate complete: publish it
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        __threadfence();
                        named_bar(2, 128);
                        if (lead)
                            mbar_arrive(&m->phik_stored[j % NPH]);
                        const int gi = r.tA / p.BH;
                        // agg_pub[j & 1] is re-armed only after the look-back warps
                        // consumed it for segment j-2 (their sin_ready follows that)
                        if (!group_ok(!lead || (bwait(&m->dseg_done, nsegA & 1, abort) &&
                                                (j < 2 || bwait(&m->sin_ready[(j - 2) & 1],
                                                                ((j - 2) >> 1) & 1, abort))),
                                      2, 128)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        float* agg =
                            p.slots + (static_cast<size_t>(r.gA.s) * p.R + gi % p.R) * kSlotFloats;
                        if (wb < 2) {  // dS^T rows = tensor-memory lanes 0..63
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t rr[16];
                                tmem_ld16(tm + TM_DSEG + lane_off + 16 * q, rr);
                                tmem_ld_wait();
                                float4* d4 = reinterpret_cast<float4*>(agg + tb * kD + 16 * q);
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    __stcg(d4 + u, make_float4(__uint_as_float(rr[4 * u]),
                                                               __uint_as_float(rr[4 * u + 1]),
                                                               __uint_as_float(rr[4 * u + 2]),
                                                               __uint_as_float(rr[4 * u + 3])));
                            }
                        } else {
                            __stcg(agg + kD * kD + (tb - 64), m->dzacc[tb - 64]);
                            m->dzacc[tb - 64] = 0.f;
                        }
                        tc_fence_before();
                        named_bar(2, 128);
                        if (lead) {
                            mbar_arrive(&m->dseg_free);
                            __threadfence();
                            st_release(p.flags + static_cast<size_t>(r.gA.s) * p.R + gi % p.R,
                                       (static_cast<unsigned>(gi + 1) << 2) | 1u);
                            mbar_arrive(&m->agg_pub[j & 1]);
                        }
                        ++nsegA;
                    }
                }
                if (k < r.nC) {  // phase C: S_prev, z_prev of chunk ci
                    const int b = ci & 1;
                    if (!group_ok(!lead || ci < 2 ||
                                      (bwait(&m->o_done[b], ((ci >> 1) & 1) ^ 1, abort) &&
                                       bwait(&m->epi_done[b], ((ci >> 1) & 1) ^ 1, abort)),
                                  2, 128) ||
                        !group_ok(!lead || ci < 1 ||
                                      bwait(&m->mma1_done[(ci - 1) & 1], ((ci - 1) >> 1) & 1,
                                            abort),
                                  2, 128) ||
                        !group_ok(!lead || k > 0 ||
                                      bwait(&m->sin_ready[jc & 1], (jc >> 1) & 1, abort),
                                  2, 128)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    unsigned char* sShi = sm + OFF_S + b * 16384;
                    unsigned char* sSlo = sShi + 8192;
                    if (wb < 2) {  // S_prev^T row tb: tensor-memory lane tb
                        float sp[kD];
                        if (k == 0) {  // segment start: S_in from the look-back
                            const float4* src = reinterpret_cast<const float4*>(
                                p.sin_scratch +
                                (static_cast<size_t>(blockIdx.x) * 2 + (jc & 1)) * kStateFloats +
                                tb * kD);
#pragma unroll
                            for (int u = 0; u < 16; ++u) {
                                const float4 x = __ldcg(src + u);
                                sp[4 * u] = x.x, sp[4 * u + 1] = x.y, sp[4 * u + 2] = x.z,
                                       sp[4 * u + 3] = x.w;
                            }
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t rr[16];
#pragma unroll
                                for (int u = 0; u < 16; ++u)
                                    rr[u] = __float_as_uint(sp[16 * q + u]);
                                tmem_st16(tm + TM_SRUN + lane_off + 16 * q, rr);
                            }
                            tmem_st_wait();
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t rr[16];
                                tmem_ld16(tm + TM_SRUN + lane_off + 16 * q, rr);
                                tmem_ld_wait();
#pragma unroll
                                for (int u = 0; u < 16; ++u)
                                    sp[16 * q + u] = __uint_as_float(rr[u]);
                            }
                        }
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc) {
                            uint4 h, l;
                            split2(sp[8 * cc + 0], sp[8 * cc + 1], h.x, l.x);
                            split2(sp[8 * cc + 2], sp[8 * cc + 3], h.y, l.y);
                            split2(sp[8 * cc + 4], sp[8 * cc + 5], h.z, l.z);
                            split2(sp[8 * cc + 6], sp[8 * cc + 7], h.w, l.w);
                            *reinterpret_cast<uint4*>(sShi + sw128_off(tb, cc)) = h;
                            *reinterpret_cast<uint4*>(sSlo + sw128_off(tb, cc)) = l;
                        }
                    } else {  // z_prev
                        const int i = tb - 64;
                        float z;
                        if (k == 0)
                            z = __ldcg(p.sin_scratch +
                                       (static_cast<size_t>(blockIdx.x) * 2 + (jc & 1)) *
                                           kStateFloats +
                                       kD * kD + i);
                        else
                            z = m->zrun[i] + m->dzk[jc % NPH][k - 1][i];
                        m->zrun[i] = z;
                        m->zprev[b][i] = z;
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    named_bar(2, 128);
                    if (lead) {
                        if (k == 0)
                            mbar_arrive(&m->sin_free[jc & 1]);
                        mbar_arrive(&m->srun_read[b]);
                        TC_TRACE(ci, 4);
                    }
                    ++ci, ++kvi;
                }
            }
            h2 = h1;
            h1 = tA;
        }
    } else if (warp >= 12) {
        // ----------------------------------------- phi(Q) (warps 12-15) ----
        const int tcx = tid - 384;
        const bool lead = tcx == 0;
        int ci = 0, h1 = -1, h2 = -1;
        bool ok = true, doneA = false;
        for (int j = 0; ok; ++j) {
            int tA = -1;
            if (!doneA) {
                if (!group_ok(!lead || bwait(&m->seg_full[j % NS], (j / NS) & 1, abort), 3, 128))
                    break;
                const int t = m->seg_ticket[j % NS];
                if (t < p.total)
                    tA = t;
                else
                    doneA = true;
            }
            Round r;
            round_setup(p, r, j, tA, h2);
            if (r.nA == 0 && r.nC == 0 && h1 < 0)
                break;
            for (int k = 0; k < r.nC; ++k, ++ci) {
                const int qs = ci % NQ;
                if (!group_ok(!lead || bwait(&m->q_full[qs], (ci / NQ) & 1, abort), 3, 128)) {
                    ok = false;
                    break;
                }
                if (lead)
                    TC_TRACE(ci, 12);
                phi_tile(sm + OFF_Q + qs * 16384, tcx, chunk_valid(p, r.gC.c0 + k), elu, nullptr,
                         nullptr);
                fence_proxy_async_smem();
                named_bar(3, 128);
                if (lead) {
                    mbar_arrive(&m->q_phi[qs]);
                    TC_TRACE(ci, 1);
                }
            }
            h2 = h1;
            h1 = tA;
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && m->abort)
        set_status(p.status, LA_ERR_TIMEOUT);
    if (warp == 0)
        tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ host --
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esz, int64_t cols,
              int64_t rows, int64_t depth, uint32_t box_cols)
{
    auto enc = encoder();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)depth};
    cuuint64_t strides[2] = {(cuuint64_t)(cols * esz), (cuuint64_t)(cols * rows * esz)};
    cuuint32_t box[3] = {box_cols, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcGeom {
    int G;       // CTAs
    int L;       // chunks per segment
    int nchunk;
    int nseg;
    int R;       // ring slots per sequence
    int total;   // segment tickets
    size_t flags_off, slots_off, sin_off, phi_off, bytes;
};

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

TcGeom tc_geom(int64_t BH, int64_t N, int sms)
{
    TcGeom g{};
    if (sms <= 0)
        sms = 148;
    g.nchunk = (int)((N + kC - 1) / kC);
    const int64_t chunks = BH * g.nchunk;
    // about a dozen segments per CTA keeps the tail short; long segments make
    // the look-back rare
    g.L = (int)std::max<int64_t>(1, std::min<int64_t>(kMaxL, chunks / ((int64_t)sms * 12)));
    g.nseg = (g.nchunk + g.L - 1) / g.L;
    g.total = (int)(BH * g.nseg);
    int G = sms;
    G = (int)std::min<int64_t>(G, g.total);
    G = (int)std::min<int64_t>(G, BH * 20);  // bounds the ring and the look-back list
    if (G < 1)
        G = 1;
    g.G = G;
    // segment tickets a CTA holds at once: the ring plus one being placed
    const int64_t per_seq = ((NS + 1) * (int64_t)G + BH - 1) / BH + 2;
    g.R = (int)std::min<int64_t>(per_seq, g.nseg);
    g.flags_off = 256;
    g.slots_off = (g.flags_off + sizeof(unsigned) * (size_t)BH * g.R + 255) & ~(size_t)255;
    g.sin_off = g.slots_off + sizeof(float) * (size_t)BH * g.R * kSlotFloats;
    g.phi_off = (g.sin_off + sizeof(float) * (size_t)G * 2 * kStateFloats + 1023) & ~(size_t)1023;
    g.bytes = g.phi_off + (size_t)G * NPH * g.L * kC * kD * 2;
    return g;
}

}  // namespace

bool tc_forward_eligible(const FwdArgs& a)
{
    return a.dtype == LA_BF16 && a.d == 64 && a.dv == 64 && a.causal == 1 && !a.gamma->has_decay &&
           a.N >= 1 && a.N <= (int64_t)INT32_MAX - kC;
}

size_t tc_forward_workspace(int64_t BH, int64_t N)
{
    return tc_geom(BH, N, sm_count()).bytes;
}

cudaError_t tc_forward(const FwdArgs& a)
{
    const int64_t BH = a.B * a.H;
    const TcGeom g = tc_geom(BH, a.N, sm_count());
    if (a.ws_bytes < g.bytes)
        return cudaErrorInvalidValue;
    TcParams p;
    memset(&p, 0, sizeof p);
    if (!make_map(&p.mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, a.N, BH, 64) ||
        !make_map(&p.mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, a.N, BH, 64) ||
        !make_map(&p.mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, a.N, BH, 64) ||
        !make_map(&p.mo, a.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 64, a.N, BH, 32))
        return cudaErrorInvalidValue;
    unsigned char* ws = static_cast<unsigned char*>(a.ws);
    if (!make_map(&p.mphi, ws + g.phi_off, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, kC,
                  (int64_t)g.G * NPH * g.L, 64))
        return cudaErrorInvalidValue;
    p.N = a.N;
    p.BH = (int)BH;
    p.nchunk = g.nchunk;
    p.L = g.L;
    p.nseg = g.nseg;
    p.R = g.R;
    p.total = g.total;
    p.fm = a.fm;
    p.counter = reinterpret_cast<unsigned*>(ws);
    p.flags = reinterpret_cast<unsigned*>(ws + g.flags_off);
    p.slots = reinterpret_cast<float*>(ws + g.slots_off);
    p.sin_scratch = reinterpret_cast<float*>(ws + g.sin_off);
    p.phi_scratch = ws + g.phi_off;
    p.status = a.status;
    cudaError_t e = cudaMemsetAsync(ws, 0, g.slots_off, a.stream);
    if (e != cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(k_fwd_tc64, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    k_fwd_tc64<<<g.G, kThreads, SMEM_BYTES, a.stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

#ifdef LA_TC_TRACE
extern "C" __attribute__((visibility("default"))) int la_debug_set_tc_trace(void* buf)
{
    return (int)cudaMemcpyToSymbol(g_tc_trace, &buf, sizeof(buf));
}
#endif

}  // namespace la
