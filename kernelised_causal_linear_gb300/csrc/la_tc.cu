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
// One persistent CTA (128 threads, two per SM) takes chunks in ticket order
// (chunk-major over the B*H sequences).  The state entering a chunk comes
// from a decoupled look-back over a small ring of per-chunk slots in global
// memory (it stays in L2): each chunk publishes its aggregate (dS_c, dz_c) as
// soon as its first MMAs finish, then its inclusive prefix.  The look-back
// starts from the nearest inclusive prefix and adds the later aggregates in
// chunk order, so every prefix is the same left-to-right fp32 sum whatever
// the timing: results are bitwise reproducible.
//
// Precision: phi(Q), phi(K) and V enter the MMAs as bf16 (phi rounded once);
// P and S_prev are fp32 and enter as a bf16 hi/lo pair (two MMAs each), so
// their rounding is ~2^-17 relative; denominators stay in fp32.
//
// Operands: Q, K, V chunks arrive by TMA in the 128-byte swizzled layout.
// The scores MMA reads Q and K K-major; the chunk-state MMA reads [V | phi(K)]
// as an MN-major A of 128 rows (the second 64 rows are discarded) against
// phi(K) MN-major, giving dS^T in lanes 0..63; P is re-packed in tensor
// memory as bf16 hi/lo and fed as the A operand of P V; S_prev^T hi/lo sit in
// shared memory K-major for phi(Q) S_prev.  The output tile is staged in
// shared memory and written by TMA.
//
// Every wait is bounded (mbarrier polls, look-back by %globaltimer); on
// expiry the CTA records LA_ERR_TIMEOUT, drains its own async work, frees its
// tensor memory and exits.
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
constexpr int kThreads = 128;
constexpr int kStateFloats = kD * kD + kD;         // S^T (dv x d) then z (d)
constexpr int kSlotFloats = 2 * kStateFloats;      // aggregate, inclusive
constexpr int kMaxList = 128;                      // look-back entries
constexpr uint32_t kPollLimit = 1u << 26;          // mbarrier polls
constexpr uint64_t kLookbackNs = 2000000000ull;    // 2 s

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;          // 128 x 64 bf16, SW128
constexpr uint32_t OFF_V = 16384;      // V directly before K: [V | K] is one
constexpr uint32_t OFF_K = 32768;      //   MN-major A with LBO = 16384
constexpr uint32_t OFF_SHI = 49152;    // S_prev^T hi, 64 x 64 bf16, SW128
constexpr uint32_t OFF_SLO = 57344;    // S_prev^T lo
constexpr uint32_t OFF_O = 65536;      // output staging, 2 x (128 x 32 fp32)
constexpr uint32_t OFF_MISC = 98304;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 2048 + 1024;  // + alignment slack

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
    uint64_t bar[5];      // kv_full, q_full, mma1, mma2, mma3
    uint32_t tmem;
    int ticket;
    int next;
    int nlist;
    int abort;
    int pad[3];
    int list[kMaxList];
    alignas(16) float zprev[kD];
    float dzpart[4][kD];
};
static_assert(sizeof(Misc) <= 2048, "misc");

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

__device__ void issue_loads(const TcParams& p, unsigned char* sm, Misc* ms, int ticket,
                            bool kv, bool q, uint64_t pol)
{
    const int c = ticket / p.BH, s = ticket % p.BH;
    if (kv) {
        mbar_arrive_expect_tx(&ms->bar[0], 2 * kC * kD * 2);
        tma_load_3d(sm + OFF_K, &p.mk, 0, c * kC, s, &ms->bar[0], pol);
        tma_load_3d(sm + OFF_V, &p.mv, 0, c * kC, s, &ms->bar[0], pol);
    }
    if (q) {
        mbar_arrive_expect_tx(&ms->bar[1], kC * kD * 2);
        tma_load_3d(sm + OFF_Q, &p.mq, 0, c * kC, s, &ms->bar[1], pol);
    }
}

__global__ void __launch_bounds__(kThreads, 2) k_fwd_tc64(const __grid_constant__ TcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Misc* ms = reinterpret_cast<Misc*>(sm + OFF_MISC);
    unsigned char* sQ = sm + OFF_Q;
    unsigned char* sK = sm + OFF_K;
    unsigned char* sV = sm + OFF_V;
    unsigned char* sShi = sm + OFF_SHI;
    unsigned char* sSlo = sm + OFF_SLO;
    unsigned char* sO = sm + OFF_O;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool norm = p.fm != LA_FM_NONE;
    const bool elu = p.fm == LA_FM_ELU1;
    const uint64_t pol = policy_evict_first();

    if (tid == 0) {
        for (int i = 0; i < 5; ++i)
            mbar_init(&ms->bar[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&p.mq);
        tma_prefetch_desc(&p.mk);
        tma_prefetch_desc(&p.mv);
        tma_prefetch_desc(&p.mo);
        ms->abort = 0;
        const int t = (int)atomicAdd(p.counter, 1u);
        ms->ticket = t;
        if (t < p.total)
            issue_loads(p, sm, ms, t, true, true, pol);
    }
    if (warp == 0) {
        tmem_alloc(&ms->tmem, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = ms->tmem;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tP = tm + lane_off;          // cols [0,128): scores / P hi,lo
    const uint32_t tO = tm + 128 + lane_off;    // cols [128,192): output
    const uint32_t tS = tm + 192 + lane_off;    // cols [192,256): dS^T (lanes 0..63)

    // Each barrier completes once per chunk; ph is the parity of the current
    // chunk.  Thread 0 tracks what is still in flight for the drain on abort.
    bool kv_pending = ms->ticket < p.total, q_pending = kv_pending;
    uint32_t kv_par = 0, q_par = 0;  // parity of the next completion of bar[0] / bar[1]
    int mma_bar = -1;                // last committed MMA barrier not yet waited on
    uint32_t mma_par = 0;
    uint32_t ph = 0;

    for (;;) {
        const int ticket = ms->ticket;
        if (ticket >= p.total)
            break;
        const int c = ticket / p.BH, s = ticket % p.BH;
        const int64_t t0 = static_cast<int64_t>(c) * kC;
        const int valid = static_cast<int>(min(static_cast<int64_t>(kC), p.N - t0));
        float* slot_base = p.slots + static_cast<size_t>(s) * p.R * kSlotFloats;
        unsigned* flag_base = p.flags + static_cast<size_t>(s) * p.R;
        const int my_slot = c % p.R;

        if (tid == 0) {  // prefetch the next ticket: its K,V load overlaps this chunk
            const int t = (int)atomicAdd(p.counter, 1u);
            ms->next = t;
        }
        bool ok = mbar_wait(&ms->bar[0], kv_par, kPollLimit);
        if (ok) {
            kv_pending = false;
            kv_par ^= 1u;
            ok = mbar_wait(&ms->bar[1], q_par, kPollLimit);
            if (ok) {
                q_pending = false;
                q_par ^= 1u;
            }
        }
        if (!ok)
            atomicExch(&ms->abort, 1);
        if (tid == 0)
            bulk_wait_read<0>();  // the previous output tile has left the staging buffer

        // ---- feature map in place, ragged rows zeroed, column sums of phi(K)
        {
            const int cc = tid & 7;
            float zp[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                zp[e] = 0.f;
#pragma unroll 2
            for (int m = 0; m < 8; ++m) {
                const int r = (tid >> 3) + 16 * m;
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
                    ms->dzpart[warp][8 * cc + e] = zp[e];
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (ms->abort)
            break;

        // ---- MMA 1: scores and chunk state
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_sc = idesc_bf16_f32(128, 128, false, false);
            const uint32_t id_st = idesc_bf16_f32(128, 64, true, true);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tm, sdesc_sw128(smem_addr(sQ) + 32 * k, 16, 1024),
                            sdesc_sw128(smem_addr(sK) + 32 * k, 16, 1024), id_sc, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_bf16_ss(tm + 192, sdesc_sw128(smem_addr(sV) + 2048 * k, OFF_K - OFF_V, 1024),
                            sdesc_sw128(smem_addr(sK) + 2048 * k, 16, 1024), id_st, k > 0);
            mma_commit(&ms->bar[2]);
            mma_bar = 2, mma_par = ph;
        }
        ok = mbar_wait(&ms->bar[2], ph, kPollLimit);
        if (ok && tid == 0)
            mma_bar = -1;
        tc_fence_after();

        // ---- dS^T (tensor-memory lanes 0..63 -> warps 0,1) and dz into a shared
        // copy (the output staging buffer is idle until the epilogue), then the
        // whole CTA writes the aggregate slot with coalesced stores
        float* sDS = reinterpret_cast<float*>(sO);  // [64][64] then z[64]
        float* agg = slot_base + static_cast<size_t>(my_slot) * kSlotFloats;
        if (warp < 2) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t r[16];
                tmem_ld16(tS + 16 * q, r);
                tmem_ld_wait();
                float4* d4 = reinterpret_cast<float4*>(sDS + tid * kD + 16 * q);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    d4[u] = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                        __uint_as_float(r[4 * u + 2]),
                                        __uint_as_float(r[4 * u + 3]));
            }
        } else {
            const int i = tid - 64;
            sDS[kD * kD + i] =
                ms->dzpart[0][i] + ms->dzpart[1][i] + ms->dzpart[2][i] + ms->dzpart[3][i];
        }
        __syncthreads();
        {
            const float4* src = reinterpret_cast<const float4*>(sDS);
            float4* dst = reinterpret_cast<float4*>(agg);
            for (int f = tid; f < kStateFloats / 4; f += kThreads)
                __stcg(dst + f, src[f]);
        }

        // ---- P: causal mask, row sums, bf16 hi/lo re-packed in place
        float den = 0.f;
        {
            uint32_t v[128];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t r[16];
                tmem_ld16(tP + 16 * q, r);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    v[16 * q + j] = r[j];
            }
            tmem_ld_wait();
            const int i = tid;  // query row within the chunk
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int j = 32 * q + 2 * m;
                    const float a = j <= i ? __uint_as_float(v[j]) : 0.f;
                    const float b = j + 1 <= i ? __uint_as_float(v[j + 1]) : 0.f;
                    den += a + b;
                    split2(a, b, hi[m], lo[m]);
                }
                tmem_st16(tP + 16 * q, hi);
                tmem_st16(tP + 64 + 16 * q, lo);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();

        // ---- flag the aggregate, MMA 2 (P V), look-back over the predecessors
        if (tid == 0) {
            __threadfence();
            st_release(flag_base + my_slot, (static_cast<unsigned>(c + 1) << 2) | 1u);
            tc_fence_after();
            const uint32_t id_pv = idesc_bf16_f32(128, 64, false, true);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_bf16_ts(tm + 128, tm + 8 * k,
                            sdesc_sw128(smem_addr(sV) + 2048 * k, 16, 1024), id_pv, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_bf16_ts(tm + 128, tm + 64 + 8 * k,
                            sdesc_sw128(smem_addr(sV) + 2048 * k, 16, 1024), id_pv, 1);
            mma_commit(&ms->bar[3]);
            mma_bar = 3, mma_par = ph;
        }
        if (warp == 0) {
            // Lane l watches chunk base - l.  The list collects, newest first, the
            // aggregates back to the nearest inclusive prefix (or the sequence start).
            // Window of W lanes: with a wrapping ring only R-1 slots behind this
            // chunk are distinct from its own.  A slot that holds another epoch
            // (older: not yet written; newer: reused after a later inclusive
            // prefix made it unnecessary) reads as not ready.
            const int W = p.R >= p.nchunk ? 32 : min(32, p.R - 1);
            const unsigned active = W >= 32 ? 0xffffffffu : ((1u << W) - 1u);
            int n = 0;
            int base = c - 1;
            uint64_t start = 0;
            const unsigned full = 0xffffffffu;
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
                            ms->list[n + lane] = (pc % p.R) << 1;
                        if (lane == ls && pc >= 0)
                            ms->list[n + lane] = ((pc % p.R) << 1) | 1;
                        n += ls + (base - ls >= 0 ? 1 : 0);
                        break;
                    }
                } else if (mr == active) {
                    if (n + W > kMaxList) {
                        n = -2;
                        break;
                    }
                    if (lane < W)
                        ms->list[n + lane] = (pc % p.R) << 1;
                    n += W;
                    base -= W;
                    start = 0;
                    continue;
                }
                const uint64_t now = globaltimer();
                if (!start)
                    start = now;
                else if (now - start > kLookbackNs) {
                    n = -1;
                    break;
                }
                __nanosleep(64);
            }
            if (lane == 0) {
                ms->nlist = n;
                if (n < 0)
                    set_status(p.status, n == -1 ? LA_ERR_TIMEOUT : LA_ERR_DEVICE_CHECK);
                // K, V are free once P V is done: start the next chunk's K, V
                if (mbar_wait(&ms->bar[3], ph, kPollLimit)) {
                    mma_bar = -1;
                    if (ms->next < p.total) {
                        issue_loads(p, sm, ms, ms->next, true, false, pol);
                        kv_pending = true;
                    }
                } else {
                    ms->nlist = -1;
                    set_status(p.status, LA_ERR_TIMEOUT);
                }
            }
        }
        __syncthreads();
        const int nlist = ms->nlist;
        if (nlist < 0 || !ok) {
            atomicExch(&ms->abort, 1);
            break;
        }

        // ---- S_prev, z_prev: the nearest inclusive prefix plus the later
        // aggregates in chunk order (a fixed left-to-right fp32 sum).  Thread t
        // owns float4 words t + 128 m of the state; threads 0..15 also z.
        {
            float4 acc[9];
#pragma unroll
            for (int m = 0; m < 9; ++m)
                acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int e = nlist - 1; e >= 0; --e) {
                const int ent = ms->list[e];
                const float4* src = reinterpret_cast<const float4*>(
                    slot_base + static_cast<size_t>(ent >> 1) * kSlotFloats +
                    ((ent & 1) ? kStateFloats : 0));
                float4 x[9];
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    x[m] = __ldcg(src + tid + 128 * m);
                x[8] = tid < 16 ? __ldcg(src + 1024 + tid) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int m = 0; m < 9; ++m) {
                    acc[m].x += x[m].x, acc[m].y += x[m].y;
                    acc[m].z += x[m].z, acc[m].w += x[m].w;
                }
            }
            const float4* ds4 = reinterpret_cast<const float4*>(sDS);
            float4* inc = reinterpret_cast<float4*>(agg + kStateFloats);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int f = tid + 128 * m;
                const int row = f >> 4, col4 = f & 15;  // S_prev^T row (value channel), 4 features
                uint2 h, l;
                split2(acc[m].x, acc[m].y, h.x, l.x);
                split2(acc[m].z, acc[m].w, h.y, l.y);
                const uint32_t off = sw128_off(row, col4 >> 1) + (col4 & 1) * 8;
                *reinterpret_cast<uint2*>(sShi + off) = h;
                *reinterpret_cast<uint2*>(sSlo + off) = l;
                const float4 d = ds4[f];
                __stcg(inc + f, make_float4(acc[m].x + d.x, acc[m].y + d.y, acc[m].z + d.z,
                                            acc[m].w + d.w));
            }
            if (tid < 16) {
                reinterpret_cast<float4*>(ms->zprev)[tid] = acc[8];
                const float4 d = ds4[1024 + tid];
                __stcg(inc + 1024 + tid, make_float4(acc[8].x + d.x, acc[8].y + d.y,
                                                     acc[8].z + d.z, acc[8].w + d.w));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- flag the inclusive prefix, MMA 3 (phi(Q) S_prev, hi and lo)
        if (tid == 0) {
            __threadfence();
            st_release(flag_base + my_slot, (static_cast<unsigned>(c + 1) << 2) | 2u);
            tc_fence_after();
            if (nlist > 0) {
                const uint32_t id_in = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16_ss(tm + 128, sdesc_sw128(smem_addr(sQ) + 32 * k, 16, 1024),
                                sdesc_sw128(smem_addr(sShi) + 32 * k, 16, 1024), id_in, 1);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16_ss(tm + 128, sdesc_sw128(smem_addr(sQ) + 32 * k, 16, 1024),
                                sdesc_sw128(smem_addr(sSlo) + 32 * k, 16, 1024), id_in, 1);
            }
            mma_commit(&ms->bar[4]);
            mma_bar = 4, mma_par = ph;
        }

        // ---- denominator: rowsum(P) + phi(q_i) . z_prev  (fp32)
        if (norm) {
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 x = *reinterpret_cast<const uint4*>(sQ + sw128_off(tid, cc));
                const float* z = ms->zprev + 8 * cc;
                den = fmaf(bf_lo(x.x), z[0], den);
                den = fmaf(bf_hi(x.x), z[1], den);
                den = fmaf(bf_lo(x.y), z[2], den);
                den = fmaf(bf_hi(x.y), z[3], den);
                den = fmaf(bf_lo(x.z), z[4], den);
                den = fmaf(bf_hi(x.z), z[5], den);
                den = fmaf(bf_lo(x.w), z[6], den);
                den = fmaf(bf_hi(x.w), z[7], den);
            }
        }
        ok = mbar_wait(&ms->bar[4], ph, kPollLimit);
        if (ok && tid == 0)
            mma_bar = -1;
        tc_fence_after();
        if (!ok)
            atomicExch(&ms->abort, 1);

        // ---- epilogue: o = num / den -> staging (SW128 fp32, two 32-column boxes)
        {
            const float inv = norm ? 1.0f / fmaxf(den, FLT_MIN) : 1.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t r[16];
                tmem_ld16(tO + 16 * q, r);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int col4 = 4 * q + u;  // 16-byte group of output columns
                    float4 o = make_float4(__uint_as_float(r[4 * u]) * inv,
                                           __uint_as_float(r[4 * u + 1]) * inv,
                                           __uint_as_float(r[4 * u + 2]) * inv,
                                           __uint_as_float(r[4 * u + 3]) * inv);
                    *reinterpret_cast<float4*>(sO + (col4 >> 3) * 16384 +
                                               sw128_off(tid, col4 & 7)) = o;
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (ms->abort)
            break;
        if (tid == 0) {
            tma_store_3d(&p.mo, sO, 0, c * kC, s, pol);
            tma_store_3d(&p.mo, sO + 16384, 32, c * kC, s, pol);
            bulk_commit();
            ms->ticket = ms->next;
            if (ms->next < p.total) {
                issue_loads(p, sm, ms, ms->next, false, true, pol);
                q_pending = true;
            }
        }
        ph ^= 1u;
        __syncthreads();
    }

    // ---- teardown (also the drain after an abort)
    if (tid == 0) {
        if (ms->abort) {
            set_status(p.status, LA_ERR_TIMEOUT);
            if (kv_pending)
                mbar_wait(&ms->bar[0], kv_par, kPollLimit);
            if (q_pending)
                mbar_wait(&ms->bar[1], q_par, kPollLimit);
            if (mma_bar >= 0)  // MMAs retire in order: the last commit covers all
                mbar_wait(&ms->bar[mma_bar], mma_par, kPollLimit);
        }
        bulk_wait<0>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(tm, 256);
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
    int G = 2 * (sms > 0 ? sms : 148);
    G = (int)std::min<int64_t>(G, g.total);
    G = (int)std::min<int64_t>(G, BH * 60);  // bounds the ring and the look-back list
    if (G < 1)
        G = 1;
    g.G = G;
    const int64_t per_seq = (2 * (int64_t)G + BH - 1) / BH + 2;  // tickets in flight / sequence
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

}  // namespace la
