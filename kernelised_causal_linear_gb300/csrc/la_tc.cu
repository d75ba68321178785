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
// Chunks are taken in ticket order (chunk-major over the B*H sequences) by one
// persistent CTA per SM.  The state entering a chunk comes from a decoupled
// look-back over a small ring of per-chunk slots in global memory (it stays in
// L2): each chunk publishes its aggregate (dS_c, dz_c) as soon as its first
// MMAs finish, then its inclusive prefix.  The look-back starts from the
// nearest inclusive prefix and adds the later aggregates in chunk order, so
// every prefix is the same left-to-right fp32 sum whatever the timing: the
// results are bitwise reproducible.
//
// The CTA is warp-specialised; chunks flow through rings of shared-memory
// stages and double-buffered tensor memory, synchronised by mbarriers:
//   warp 0      producer: tickets, TMA loads of Q and of K, V
//   warp 1      MMA issuer: scores + chunk state, P V, phi(Q) S_prev
//   warp 2      look-back over the predecessors' flags (needs only the ticket,
//               so it runs ahead of the chunk's own arithmetic)
//   warps 4-7   feature map in place, column sums of phi(K); P: causal mask,
//               row sums, bf16 hi/lo re-pack in tensor memory
//   warps 8-11  chunk state out of tensor memory, aggregate and inclusive
//               prefix publishing, S_prev hi/lo for the tensor cores
//   warps 12-15 epilogue: denominator, output tile by TMA store
//
// Precision: phi(Q), phi(K) and V enter the MMAs as bf16 (phi rounded once);
// P and S_prev are fp32 and enter as a bf16 hi/lo pair (two MMAs each), so
// their rounding is ~2^-17 relative; denominators stay in fp32.
//
// Operands: Q, K, V chunks arrive by TMA in the 128-byte swizzled layout.
// The scores MMA reads Q and K K-major; the chunk-state MMA reads [V | phi(K)]
// as an MN-major A of 128 rows (the second 64 rows are discarded) against
// phi(K) MN-major, giving dS^T in lanes 0..63; P's hi/lo parts sit in tensor
// memory as the A operand of P V; S_prev^T hi/lo sit in shared memory
// K-major for phi(Q) S_prev.
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
constexpr int NKV = 2;         // K,V stages
constexpr int NT = 4;          // ticket ring
constexpr int kStateFloats = kD * kD + kD;         // S^T (dv x d) then z (d)
constexpr int kSlotFloats = 2 * kStateFloats;      // aggregate, inclusive
constexpr int kMaxList = 128;                      // look-back entries
constexpr uint64_t kWaitNs = 2000000000ull;        // 2 s for any single wait

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;                          // NQ x (128 x 64 bf16)
constexpr uint32_t OFF_KV = OFF_Q + NQ * 16384;        // NKV x (V then K)
constexpr uint32_t OFF_S = OFF_KV + NKV * 32768;       // 2 x (S^T hi, S^T lo)
constexpr uint32_t OFF_O = OFF_S + 2 * 16384;          // output staging 2 x 16 KiB
constexpr uint32_t OFF_DS = OFF_O + 32768;             // dS^T, dz fp32 copy
constexpr uint32_t OFF_MISC = OFF_DS + 17408;
constexpr uint32_t kMiscBytes = 6144;
constexpr uint32_t SMEM_BYTES = OFF_MISC + kMiscBytes + 1024;  // + alignment slack

// tensor memory columns
constexpr uint32_t TM_P = 0;      // scores fp32, 128 columns
constexpr uint32_t TM_PHL = 128;  // P hi (128..191), P lo (192..255), bf16 pairs
constexpr uint32_t TM_O = 256;    // 2 x 64: output accumulators
constexpr uint32_t TM_DS = 384;   // 2 x 64: dS^T (lanes 0..63)

struct TcParams {
    CUtensorMap mq, mk, mv, mo;
    int64_t N;
    int BH;
    int nchunk;
    int R;        // ring slots per sequence
    int total;    // BH * nchunk
    int fm;
    unsigned* counter;
    unsigned* flags;
    float* slots;
    int* status;
};

struct Misc {
    uint64_t tick_full[NT], tick_empty[NT];
    uint64_t q_full[NQ], q_empty[NQ];
    uint64_t kv_full[NKV], kv_empty[NKV];
    uint64_t phi_done[2], mma1_done[2], p_ready[2], pv_done[2], ds_free[2], s_ready[2];
    uint64_t o_done[2], o_free[2], list_full[2], list_empty[2], epi_done[2];
    uint64_t drain;
    uint32_t tmem;
    int abort;
    int ticket[NT];
    int nlist[2];
    int list[2][kMaxList];
    float den[2][kC];
    alignas(16) float zprev[2][kD];
    float dzpart[2][4][kD];
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc");

// Optional per-chunk event timestamps (SM clock) for pipeline analysis; only
// in builds with LA_TC_TRACE defined, never in the library as shipped.
#ifdef LA_TC_TRACE
__device__ unsigned long long* g_tc_trace;
#define TC_TRACE(i, ev)                                                                  \
    do {                                                                                 \
        if (g_tc_trace && (i) < 64)                                                      \
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

__device__ __forceinline__ void named_bar(int id)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(128) : "memory");
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    uint64_t t0 = 0;
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((n & 31u) == 0u) {
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

// A 128-thread group waits through one leader; bar.red hands every thread
// the same verdict, so the group never splits on an abort.
__device__ __forceinline__ bool group_ok(int ok, int barid)
{
    int res;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.and.pred p, %2, 128, p;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(res)
        : "r"(ok), "r"(barid)
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

// elu(x)+1 on two packed bf16, rounded back to bf16
__device__ __forceinline__ uint32_t phi2(uint32_t w)
{
    float a = bf_lo(w), b = bf_hi(w);
    a = a > 0.f ? a + 1.f : __expf(a);
    b = b > 0.f ? b + 1.f : __expf(b);
    return pack_bf16x2(a, b);
}

// split two fp32 into packed bf16 hi and lo parts
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo)
{
    hi = pack_bf16x2(a, b);
    lo = pack_bf16x2(a - bf_lo(hi), b - bf_hi(hi));
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
    }
    if (warp == 0) {
        tmem_alloc(&m->tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = m->tmem;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int q_last[NQ], kv_last[NKV];
            for (int j = 0; j < NQ; ++j)
                q_last[j] = -1;
            for (int j = 0; j < NKV; ++j)
                kv_last[j] = -1;
            for (int i = 0;; ++i) {
                const int t = static_cast<int>(atomicAdd(p.counter, 1u));
                const int ts = i % NT;
                if (i >= NT && !bwait(&m->tick_empty[ts], ((i / NT) & 1) ^ 1, abort))
                    break;
                m->ticket[ts] = t;
                mbar_arrive(&m->tick_full[ts]);
                TC_TRACE(i, 0);
                if (t >= p.total)
                    break;
                const int c = t / p.BH, s = t % p.BH;
                const int qs = i % NQ, ks = i % NKV;
                if (i >= NQ && !bwait(&m->q_empty[qs], ((i / NQ) & 1) ^ 1, abort))
                    break;
                mbar_arrive_expect_tx(&m->q_full[qs], kC * kD * 2);
                tma_load_3d(sm + OFF_Q + qs * 16384, &p.mq, 0, c * kC, s, &m->q_full[qs], pol);
                q_last[qs] = i / NQ;
                TC_TRACE(i, 1);
                if (i >= NKV && !bwait(&m->kv_empty[ks], ((i / NKV) & 1) ^ 1, abort))
                    break;
                mbar_arrive_expect_tx(&m->kv_full[ks], 2 * kC * kD * 2);
                unsigned char* kv = sm + OFF_KV + ks * 32768;
                tma_load_3d(kv + 16384, &p.mk, 0, c * kC, s, &m->kv_full[ks], pol);
                tma_load_3d(kv, &p.mv, 0, c * kC, s, &m->kv_full[ks], pol);
                kv_last[ks] = i / NKV;
                TC_TRACE(i, 2);
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
            bool issued = false;
            // MMA 1 of chunk i: scores into TM_P, chunk state into TM_DS[b]
            auto mma1 = [&](int i) -> int {  // 1 issued, 0 no such chunk, -1 abort
                const int ts = i % NT;
                if (!bwait(&m->tick_full[ts], (i / NT) & 1, abort))
                    return -1;
                if (m->ticket[ts] >= p.total)
                    return 0;
                const int b = i & 1;
                if (!bwait(&m->phi_done[b], (i >> 1) & 1, abort))
                    return -1;
                if (i >= 2 && !bwait(&m->ds_free[b], ((i >> 1) & 1) ^ 1, abort))
                    return -1;
                tc_fence_after();
                const uint32_t q = smem_addr(sm + OFF_Q + (i % NQ) * 16384);
                const uint32_t v = smem_addr(sm + OFF_KV + (i % NKV) * 32768);
                const uint32_t k = v + 16384;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tm + TM_P, sdesc_sw128(q + 32 * kk, 16, 1024),
                                sdesc_sw128(k + 32 * kk, 16, 1024), id_sc, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ss(tm + TM_DS + 64 * b, sdesc_sw128(v + 2048 * kk, 16384, 1024),
                                sdesc_sw128(k + 2048 * kk, 16, 1024), id_st, kk > 0);
                mma_commit(&m->mma1_done[b]);
                TC_TRACE(i, 7);
                issued = true;
                return 1;
            };
            int r = mma1(0);
            for (int i = 0; r == 1; ++i) {
                const int b = i & 1;
                if (!bwait(&m->p_ready[b], (i >> 1) & 1, abort))
                    break;
                if (i >= 2 && !bwait(&m->o_free[b], ((i >> 1) & 1) ^ 1, abort))
                    break;
                tc_fence_after();
                const uint32_t v = smem_addr(sm + OFF_KV + (i % NKV) * 32768);
                const uint32_t o = tm + TM_O + 64 * b;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(o, tm + TM_PHL + 8 * kk, sdesc_sw128(v + 2048 * kk, 16, 1024),
                                id_pv, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(o, tm + TM_PHL + 64 + 8 * kk,
                                sdesc_sw128(v + 2048 * kk, 16, 1024), id_pv, 1);
                mma_commit(&m->pv_done[b]);
                mma_commit(&m->kv_empty[i % NKV]);
                TC_TRACE(i, 8);
                r = mma1(i + 1);
                if (r < 0)
                    break;
                if (!bwait(&m->s_ready[b], (i >> 1) & 1, abort))
                    break;
                tc_fence_after();
                const uint32_t q = smem_addr(sm + OFF_Q + (i % NQ) * 16384);
                const uint32_t sh = smem_addr(sm + OFF_S + b * 16384);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(o, sdesc_sw128(q + 32 * kk, 16, 1024),
                                sdesc_sw128(sh + 32 * kk, 16, 1024), id_in, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(o, sdesc_sw128(q + 32 * kk, 16, 1024),
                                sdesc_sw128(sh + 8192 + 32 * kk, 16, 1024), id_in, 1);
                mma_commit(&m->o_done[b]);
                TC_TRACE(i, 9);
            }
            if (issued && *abort) {  // every MMA issued here retires before tensor memory is freed
                mma_commit(&m->drain);
                drain_wait(&m->drain, 0);
            }
        }
    } else if (warp == 2) {
        // ----------------------------------------------------- look-back --
        const unsigned full = 0xffffffffu;
        for (int i = 0;; ++i) {
            const int ts = i % NT;
            int ok = 1;
            if (lane == 0)
                ok = bwait(&m->tick_full[ts], (i / NT) & 1, abort);
            if (!__shfl_sync(full, ok, 0))
                break;
            const int t = m->ticket[ts];
            if (t >= p.total)
                break;
            const int b = i & 1;
            if (lane == 0 && i >= 2)
                ok = bwait(&m->list_empty[b], ((i >> 1) & 1) ^ 1, abort);
            if (!__shfl_sync(full, ok, 0))
                break;
            const int c = t / p.BH, s = t % p.BH;
            if (lane == 0)
                TC_TRACE(i, 10);
            const unsigned* flag_base = p.flags + static_cast<size_t>(s) * p.R;
            // Lane l watches chunk base - l.  With a wrapping ring only R-1 slots
            // behind this chunk are distinct from its own; a slot that holds
            // another epoch (older: not yet written; newer: reused once a later
            // inclusive prefix made it unnecessary) reads as not ready.
            const int W = p.R >= p.nchunk ? 32 : min(32, p.R - 1);
            const unsigned active = W >= 32 ? 0xffffffffu : ((1u << W) - 1u);
            int* list = m->list[b];
            int n = 0, base = c - 1;
            uint64_t start = 0;
            while (base >= 0) {
                const int pc = base - lane;
                bool ready = true, incl = true;
                if (lane >= W) {
                    ready = incl = false;
                } else if (pc >= 0) {
                    const unsigned f = ld_acquire(flag_base + pc % p.R);
                    ready = (f >> 2) == static_cast<unsigned>(pc + 1) && (f & 3u) != 0u;
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
                            list[n + lane] = (pc % p.R) << 1;
                        if (lane == ls && pc >= 0)
                            list[n + lane] = ((pc % p.R) << 1) | 1;
                        n += ls + (base - ls >= 0 ? 1 : 0);
                        break;
                    }
                } else if (mr == active) {
                    if (n + W > kMaxList) {
                        n = -2;
                        break;
                    }
                    if (lane < W)
                        list[n + lane] = (pc % p.R) << 1;
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
                __nanosleep(32);
            }
            __syncwarp();
            if (n < 0) {
                if (lane == 0) {
                    set_status(p.status, n == -1 ? LA_ERR_TIMEOUT : LA_ERR_DEVICE_CHECK);
                    *abort = 1;
                }
                break;
            }
            if (lane == 0) {
                m->nlist[b] = n;
                mbar_arrive(&m->list_full[b]);
                TC_TRACE(i, 11);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // --------------------------------- feature map, P (warps 4-7) --
        const int ta = tid - 128, wa = warp - 4;
        const bool lead = ta == 0;
        for (int i = 0;; ++i) {
            const int ts = i % NT;
            if (!group_ok(!lead || bwait(&m->tick_full[ts], (i / NT) & 1, abort), 1))
                break;
            const int t = m->ticket[ts];
            if (t >= p.total)
                break;
            const int c = t / p.BH;
            const int valid = static_cast<int>(min(static_cast<int64_t>(kC),
                                                   p.N - static_cast<int64_t>(c) * kC));
            const int b = i & 1;
            if (!group_ok(!lead || (bwait(&m->q_full[i % NQ], (i / NQ) & 1, abort) &&
                                    bwait(&m->kv_full[i % NKV], (i / NKV) & 1, abort) &&
                                    (i < 2 || bwait(&m->ds_free[b], ((i >> 1) & 1) ^ 1, abort))),
                          1))
                break;
            unsigned char* sQ = sm + OFF_Q + (i % NQ) * 16384;
            unsigned char* sK = sm + OFF_KV + (i % NKV) * 32768 + 16384;
            if (lead)
                TC_TRACE(i, 3);
            {
                const int cc = ta & 7;
                float zp[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    zp[e] = 0.f;
#pragma unroll 2
                for (int mm = 0; mm < 8; ++mm) {
                    const int r = (ta >> 3) + 16 * mm;
                    const uint32_t off = sw128_off(r, cc);
                    uint4* pq = reinterpret_cast<uint4*>(sQ + off);
                    uint4* pk = reinterpret_cast<uint4*>(sK + off);
                    uint4 xq = *pq, xk = *pk;
                    if (r >= valid) {
                        xq = make_uint4(0, 0, 0, 0);
                        xk = make_uint4(0, 0, 0, 0);
                        *pq = xq;
                        *pk = xk;
                    } else if (elu) {
                        xq = make_uint4(phi2(xq.x), phi2(xq.y), phi2(xq.z), phi2(xq.w));
                        xk = make_uint4(phi2(xk.x), phi2(xk.y), phi2(xk.z), phi2(xk.w));
                        *pq = xq;
                        *pk = xk;
                    }
                    zp[0] += bf_lo(xk.x), zp[1] += bf_hi(xk.x);
                    zp[2] += bf_lo(xk.y), zp[3] += bf_hi(xk.y);
                    zp[4] += bf_lo(xk.z), zp[5] += bf_hi(xk.z);
                    zp[6] += bf_lo(xk.w), zp[7] += bf_hi(xk.w);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    zp[e] += __shfl_xor_sync(0xffffffffu, zp[e], 8);
                    zp[e] += __shfl_xor_sync(0xffffffffu, zp[e], 16);
                }
                if (lane < 8)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        m->dzpart[b][wa][8 * cc + e] = zp[e];
            }
            fence_proxy_async_smem();
            named_bar(1);
            if (ta == 0) {
                mbar_arrive(&m->phi_done[b]);
                TC_TRACE(i, 4);
            }

            // P: causal mask, row sums, bf16 hi/lo into TM_PHL
            if (!group_ok(!lead || (bwait(&m->mma1_done[b], (i >> 1) & 1, abort) &&
                                    (i < 1 || bwait(&m->pv_done[(i - 1) & 1],
                                                    ((i - 1) >> 1) & 1, abort)) &&
                                    (i < 2 || bwait(&m->epi_done[b], ((i >> 1) & 1) ^ 1, abort))),
                          1))
                break;
            tc_fence_after();
            if (lead)
                TC_TRACE(i, 5);
            float rs = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t v0[16], v1[16];
                tmem_ld16(tm + TM_P + lane_off + 32 * q, v0);
                tmem_ld16(tm + TM_P + lane_off + 32 * q + 16, v1);
                tmem_ld_wait();
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int mm = 0; mm < 16; ++mm) {
                    const int j = 32 * q + 2 * mm;
                    const uint32_t wa0 = mm < 8 ? v0[2 * mm] : v1[2 * mm - 16];
                    const uint32_t wa1 = mm < 8 ? v0[2 * mm + 1] : v1[2 * mm - 15];
                    const float a = j <= ta ? __uint_as_float(wa0) : 0.f;
                    const float bb = j + 1 <= ta ? __uint_as_float(wa1) : 0.f;
                    rs += a + bb;
                    split2(a, bb, hi[mm], lo[mm]);
                }
                tmem_st16(tm + TM_PHL + lane_off + 16 * q, hi);
                tmem_st16(tm + TM_PHL + lane_off + 64 + 16 * q, lo);
            }
            tmem_st_wait();
            m->den[b][ta] = rs;
            tc_fence_before();
            named_bar(1);
            if (ta == 0) {
                mbar_arrive(&m->p_ready[b]);
                TC_TRACE(i, 6);
            }
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------ chunk state, prefixes (warps 8-11) --
        const int tb = tid - 256, wb = warp - 8;
        float* sDS = reinterpret_cast<float*>(sm + OFF_DS);
        const bool lead = tb == 0;
        for (int i = 0;; ++i) {
            const int ts = i % NT;
            if (!group_ok(!lead || bwait(&m->tick_full[ts], (i / NT) & 1, abort), 2))
                break;
            const int t = m->ticket[ts];
            if (t >= p.total)
                break;
            const int c = t / p.BH, s = t % p.BH;
            const int b = i & 1;
            float* slot_base = p.slots + static_cast<size_t>(s) * p.R * kSlotFloats;
            unsigned* flag = p.flags + static_cast<size_t>(s) * p.R + (c % p.R);
            float* agg = slot_base + static_cast<size_t>(c % p.R) * kSlotFloats;
            if (!group_ok(!lead || (bwait(&m->phi_done[b], (i >> 1) & 1, abort) &&
                                    bwait(&m->mma1_done[b], (i >> 1) & 1, abort)),
                          2))
                break;
            tc_fence_after();
            if (lead)
                TC_TRACE(i, 12);
            if (wb < 2) {  // dS^T rows = tensor-memory lanes 0..63
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t r[16];
                    tmem_ld16(tm + TM_DS + 64 * b + lane_off + 16 * q, r);
                    tmem_ld_wait();
                    float4* d4 = reinterpret_cast<float4*>(sDS + tb * kD + 16 * q);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        d4[u] = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                            __uint_as_float(r[4 * u + 2]),
                                            __uint_as_float(r[4 * u + 3]));
                }
            } else {
                const int j = tb - 64;
                sDS[kD * kD + j] = m->dzpart[b][0][j] + m->dzpart[b][1][j] + m->dzpart[b][2][j] +
                                   m->dzpart[b][3][j];
            }
            tc_fence_before();
            named_bar(2);
            if (tb == 0)
                mbar_arrive(&m->ds_free[b]);
            {  // the aggregate, coalesced
                const float4* src = reinterpret_cast<const float4*>(sDS);
                float4* dst = reinterpret_cast<float4*>(agg);
                for (int f = tb; f < kStateFloats / 4; f += 128)
                    __stcg(dst + f, src[f]);
            }
            named_bar(2);
            if (tb == 0) {
                __threadfence();
                st_release(flag, (static_cast<unsigned>(c + 1) << 2) | 1u);
                TC_TRACE(i, 13);
            }

            // S_prev, z_prev: the nearest inclusive prefix plus the later
            // aggregates in chunk order; thread tb owns float4 words tb + 128 j
            // of the state, threads 0..15 also the z words.
            if (!group_ok(!lead || bwait(&m->list_full[b], (i >> 1) & 1, abort), 2))
                break;
            const int nlist = m->nlist[b];
            float4 acc[9];
#pragma unroll
            for (int j = 0; j < 9; ++j)
                acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int e = nlist - 1; e >= 0; --e) {
                const int ent = m->list[b][e];
                const float4* src = reinterpret_cast<const float4*>(
                    slot_base + static_cast<size_t>(ent >> 1) * kSlotFloats +
                    ((ent & 1) ? kStateFloats : 0));
                float4 x[9];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    x[j] = __ldcg(src + tb + 128 * j);
                x[8] = tb < 16 ? __ldcg(src + 1024 + tb) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 9; ++j) {
                    acc[j].x += x[j].x, acc[j].y += x[j].y;
                    acc[j].z += x[j].z, acc[j].w += x[j].w;
                }
            }
            if (!group_ok(!lead || i < 2 ||
                              (bwait(&m->o_done[b], ((i >> 1) & 1) ^ 1, abort) &&
                               bwait(&m->epi_done[b], ((i >> 1) & 1) ^ 1, abort)),
                          2))
                break;
            unsigned char* sShi = sm + OFF_S + b * 16384;
            unsigned char* sSlo = sShi + 8192;
            const float4* ds4 = reinterpret_cast<const float4*>(sDS);
            float4* inc = reinterpret_cast<float4*>(agg + kStateFloats);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int f = tb + 128 * j;
                const int row = f >> 4, col4 = f & 15;  // S_prev^T row, 4 features
                uint2 h, l;
                split2(acc[j].x, acc[j].y, h.x, l.x);
                split2(acc[j].z, acc[j].w, h.y, l.y);
                const uint32_t off = sw128_off(row, col4 >> 1) + (col4 & 1) * 8;
                *reinterpret_cast<uint2*>(sShi + off) = h;
                *reinterpret_cast<uint2*>(sSlo + off) = l;
                const float4 d = ds4[f];
                __stcg(inc + f, make_float4(acc[j].x + d.x, acc[j].y + d.y, acc[j].z + d.z,
                                            acc[j].w + d.w));
            }
            if (tb < 16) {
                reinterpret_cast<float4*>(m->zprev[b])[tb] = acc[8];
                const float4 d = ds4[1024 + tb];
                __stcg(inc + 1024 + tb, make_float4(acc[8].x + d.x, acc[8].y + d.y,
                                                    acc[8].z + d.z, acc[8].w + d.w));
            }
            fence_proxy_async_smem();
            named_bar(2);
            if (tb == 0) {
                mbar_arrive(&m->list_empty[b]);
                mbar_arrive(&m->s_ready[b]);
                __threadfence();
                st_release(flag, (static_cast<unsigned>(c + 1) << 2) | 2u);
                TC_TRACE(i, 14);
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------ epilogue (warps 12-15) --
        const int tcx = tid - 384;
        const uint64_t pol = policy_evict_first();
        unsigned char* sO = sm + OFF_O;
        const bool lead = tcx == 0;
        for (int i = 0;; ++i) {
            const int ts = i % NT;
            if (!group_ok(!lead || bwait(&m->tick_full[ts], (i / NT) & 1, abort), 3))
                break;
            const int t = m->ticket[ts];
            if (t >= p.total)
                break;
            const int c = t / p.BH, s = t % p.BH;
            const int b = i & 1, qs = i % NQ;
            if (!group_ok(!lead || (bwait(&m->p_ready[b], (i >> 1) & 1, abort) &&
                                    bwait(&m->s_ready[b], (i >> 1) & 1, abort) &&
                                    bwait(&m->o_done[b], (i >> 1) & 1, abort)),
                          3))
                break;
            tc_fence_after();
            float den = 0.f;
            if (norm) {
                den = m->den[b][tcx];
                const unsigned char* sQ = sm + OFF_Q + qs * 16384;
                const float* z = m->zprev[b];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 x = *reinterpret_cast<const uint4*>(sQ + sw128_off(tcx, cc));
                    const float* zz = z + 8 * cc;
                    den = fmaf(bf_lo(x.x), zz[0], den);
                    den = fmaf(bf_hi(x.x), zz[1], den);
                    den = fmaf(bf_lo(x.y), zz[2], den);
                    den = fmaf(bf_hi(x.y), zz[3], den);
                    den = fmaf(bf_lo(x.z), zz[4], den);
                    den = fmaf(bf_hi(x.z), zz[5], den);
                    den = fmaf(bf_lo(x.w), zz[6], den);
                    den = fmaf(bf_hi(x.w), zz[7], den);
                }
            }
            const float inv = norm ? 1.0f / fmaxf(den, FLT_MIN) : 1.0f;
            if (tcx == 0)
                bulk_wait_read<0>();  // the previous tile has left the staging buffer
            named_bar(3);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t r[16];
                tmem_ld16(tm + TM_O + 64 * b + lane_off + 16 * q, r);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int col4 = 4 * q + u;
                    const float4 o = make_float4(__uint_as_float(r[4 * u]) * inv,
                                                 __uint_as_float(r[4 * u + 1]) * inv,
                                                 __uint_as_float(r[4 * u + 2]) * inv,
                                                 __uint_as_float(r[4 * u + 3]) * inv);
                    *reinterpret_cast<float4*>(sO + (col4 >> 3) * 16384 +
                                               sw128_off(tcx, col4 & 7)) = o;
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar(3);
            if (tcx == 0) {
                mbar_arrive(&m->o_free[b]);
                mbar_arrive(&m->q_empty[qs]);
                mbar_arrive(&m->epi_done[b]);
                mbar_arrive(&m->tick_empty[ts]);
                tma_store_3d(&p.mo, sO, 0, c * kC, s, pol);
                tma_store_3d(&p.mo, sO + 16384, 32, c * kC, s, pol);
                bulk_commit();
                TC_TRACE(i, 15);
            }
        }
        if (tcx == 0)
            bulk_wait<0>();
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
    int R;       // ring slots per sequence
    int nchunk;
    int total;
    size_t flags_off, slots_off, bytes;
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
    g.nchunk = (int)((N + kC - 1) / kC);
    g.total = (int)(BH * g.nchunk);
    int G = sms > 0 ? sms : 148;
    G = (int)std::min<int64_t>(G, g.total);
    G = (int)std::min<int64_t>(G, BH * 20);  // bounds the ring and the look-back list
    if (G < 1)
        G = 1;
    g.G = G;
    // tickets a CTA holds at once: the ring plus one being placed
    const int64_t per_seq = ((NT + 1) * (int64_t)G + BH - 1) / BH + 2;
    g.R = (int)std::min<int64_t>(per_seq, g.nchunk);
    g.flags_off = 256;
    g.slots_off = (g.flags_off + sizeof(unsigned) * (size_t)BH * g.R + 255) & ~(size_t)255;
    g.bytes = g.slots_off + sizeof(float) * (size_t)BH * g.R * kSlotFloats;
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
    p.N = a.N;
    p.BH = (int)BH;
    p.nchunk = g.nchunk;
    p.R = g.R;
    p.total = g.total;
    p.fm = a.fm;
    p.counter = reinterpret_cast<unsigned*>(ws);
    p.flags = reinterpret_cast<unsigned*>(ws + g.flags_off);
    p.slots = reinterpret_cast<float*>(ws + g.slots_off);
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
