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
//   [num | den] = P [V_c | 1] + phi(Q_c) [S_prev | z_prev] (tensor cores)
//   o     = num / max(den, FLT_MIN)
//   dS_c  = phi(K_c)^T V_c,  dz_c = column sums of phi(K_c)
//
// ("Linear Attention Kernel", section "Rewrite: associativity": phi(K)^T V
// is the only intermediate; "Efficient Attention Variants", section 5: the
// prefix state S_t, z_t and the normalised read).  The ones column of
// [V_c | 1] makes the row sums of P, and the extra column z_prev of the state
// operand makes phi(q).z_prev, in the same accumulator as the numerator.
//
// Chunks are grouped into segments of L consecutive chunks of one sequence.
// One persistent CTA per SM takes segments in ticket order (segment-major over
// the B*H sequences) and runs each in two phases, one round apart:
//   A  K, V of every chunk (V kept in L2 with an evict-last hint); phi(K), also
//      copied to a scratch ring for phase C; the segment's [dS^T; dz] summed
//      on the tensor cores; the total (the aggregate) is published to a ring of
//      per-segment slots in global memory;
//   C  the outputs, by the output group that owns the segment: Q, phi(K)
//      (scratch) and V (L2); S_prev of the first chunk is S_in, and after each
//      chunk but the last the chunk's [dS^T; dz] is added to the group's
//      S_prev operand in place.
// Between them a decoupled look-back over the predecessors' slots gives S_in,
// the state before the segment, and publishes it as the segment's exclusive
// prefix.  It adds the nearest exclusive prefix, that segment's aggregate and
// the later aggregates farthest first, so every prefix is the same
// left-to-right fp32 sum whatever the timing: results are bitwise
// reproducible.
//
// [V | e] (V and a constant 2 KiB block e whose first column is all ones)
// is read in two places: as the A operand of the state MMAs, where D =
// [V | e]^T phi(K) holds dS^T in lanes 0..63 and dz in lane 64, and as the B
// operand of P [V | e], whose column 64 is rowsum(P).
//
// The CTA is warp-specialised; work flows through shared-memory stages and
// tensor-memory buffers, synchronised by mbarriers:
//   warp 0      producer (one thread): segment tickets and every TMA load,
//               advancing three streams (phase A, output group 0, output
//               group 1) as their slots free up
//   warps 1-3   look-back: S_in of each segment from the predecessors'
//               slots, published as its exclusive prefix and written once as
//               the bf16 hi/lo operand image the output group loads
//   warps 4-7   phase A: phi(K) in place, copied out by TMA; the segment's
//               running [dS^T; dz] on the tensor cores; the aggregate
//   warps 8-11, 12-15
//               output groups 0 and 1, each owning every other segment:
//               phi(Q), scores, P (causal mask, bf16 hi/lo in place),
//               [num | den], epilogue (16-byte stores), then the chunk's
//               [dS^T; dz] into the S_prev operand.  Each issues its own MMAs.
//
// Precision: phi(Q), phi(K) and V enter the MMAs as bf16 (phi rounded once);
// P and S_prev are fp32 and enter as a bf16 hi/lo pair (two MMAs each), so
// their rounding is ~2^-17 relative; states and denominators stay fp32.
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
#include "la_tc_common.cuh"

namespace la {
namespace {

using namespace sm100;
using namespace tcc;

constexpr int kC = 128;        // tokens per chunk
constexpr int kD = 64;         // d = dv
constexpr int kThreads = 512;  // 16 warps
constexpr int NS = 4;          // segment-ticket ring
constexpr int NSIN = 4;        // S_in image ring (an image lives until its segment's phase C is done)
constexpr int kStateFloats = kD * kD + kD;         // S^T (dv x d) then z (d)
constexpr int kSlotFloats = 2 * kStateFloats;      // aggregate, exclusive prefix
constexpr int kMaxList = 256;                      // look-back entries
// A look-back walks over the segments of its sequence whose exclusive prefix
// is not yet out, plus two entries.  A CTA holds at most NS segment tickets
// whose phase C has not finished (the ticket ring), and a segment's prefix is
// out before its phase C starts, so at most NS such segments per CTA working
// on the sequence: 40 CTAs per sequence need at most 40 NS + 2 = 162 entries.
constexpr int kMaxCtasPerSeq = 40;
constexpr uint32_t kImgPart = 65 * 128;            // rows 0..64 of one bf16 part (hi or lo)
constexpr uint32_t kImgBytes = 2 * kImgPart;       // one state operand image: hi, then lo
constexpr uint64_t kWaitNs = 2000000000ull;        // 2 s for any single wait

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kON = 80;                                // output accumulator: num (64), den, pad
constexpr uint32_t kSBytes = kON * 128;                // [S_prev^T; z_prev] bf16, 80 x 64
constexpr int NA = 2;                                  // phase-A K,V stages
// per output warpgroup: Q, V, phi(K), [S_prev^T; z_prev] hi/lo
constexpr uint32_t CW_Q = 0, CW_V = 16384, CW_K = 32768, CW_S = 49152;
constexpr uint32_t kCWBytes = CW_S + 2 * kSBytes;
constexpr uint32_t OFF_CW = 0;                         // 2 x kCWBytes
constexpr uint32_t OFF_A = OFF_CW + 2 * kCWBytes;      // NA x (V then K)
constexpr uint32_t OFF_MISC = OFF_A + NA * 32768;
constexpr uint32_t kMiscBytes = 2048;
constexpr uint32_t OFF_ONES = OFF_MISC + kMiscBytes;   // 2 KiB: the e rows of [V | e]
constexpr int kMaxL = 8;       // largest segment (chunks)
constexpr int kMinL = 4;       // smallest segment (chunks), unless the sequence is shorter
#ifndef LA_TC_SEG_DIV
#define LA_TC_SEG_DIV 8        // segments per CTA the segment length aims at
#endif
constexpr int NPH = 4;         // phi(K) scratch ring depth, in segments
constexpr uint32_t SMEM_BYTES = OFF_ONES + 2048 + 1024;  // + alignment slack
static_assert(OFF_ONES % 1024 == 0 && kCWBytes % 1024 == 0 && kSBytes % 1024 == 0 &&
                  CW_S == CW_K + 16384 && CW_S + 16384 <= kCWBytes,
              "layout");
static_assert(SMEM_BYTES <= 232448, "shared memory");

// tensor memory columns
constexpr uint32_t TM_P = 0;       // 2 x 128: scores fp32, then P hi/lo in place
constexpr uint32_t TM_O = 256;     // 2 x 80: [num | den] accumulators
constexpr uint32_t TM_DSEG = 448;  // segment aggregate so far [dS^T; dz] (lanes 0..64)

struct TcParams {
    CUtensorMap mq, mk, mv;
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
    unsigned char* sin_img;  // per CTA: NSIN operand images of [S_in^T; z_in] (kImgBytes)
    void* phi_scratch;   // the tiles mphi describes
    float* out;          // [BH][N][64] fp32
    int* status;
};

struct Misc {
    uint64_t seg_full[NS], seg_empty[NS];
    uint64_t a_full[NA], a_empty[NA];
    uint64_t q_full[2], v_full[2], k_full[2], qs_free[2], ds_done[2], s_done[2], o_done[2];
    uint64_t phik_stored[NPH], dseg_done, sin_ready[NSIN], sin_free[NSIN], agg_ready[NSIN];
    uint64_t drain[5];
    uint32_t tmem;
    int abort;
    int seg_ticket[NS];
    int nlist;
    int list[kMaxList];
    volatile int trace_done;
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc");

// Optional per-chunk event timestamps (SM clock) for pipeline analysis; only
// in builds with LA_TC_TRACE defined, never in the library as shipped.
#ifdef LA_TC_TRACE
__device__ unsigned long long* g_tc_trace;
#define TC_TRACE(i, ev)                                                                       \
    do {                                                                                      \
        if (g_tc_trace && (i) < 64)                                                           \
            g_tc_trace[(static_cast<size_t>(blockIdx.x) * 64 + (i)) * 32 + (ev)] = clock64(); \
    } while (0)
#else
#define TC_TRACE(i, ev) \
    do {                \
    } while (0)
#endif

// Test hooks of the give-up path (la_debug_set_tc_faults): the limit of any
// single wait, and one segment ticket whose aggregate and exclusive prefix are
// never published, so that its successors' look-backs run out of time.  The
// library sets neither: 2 s and no ticket.
__device__ uint64_t g_tc_wait_ns = kWaitNs;
__device__ int g_tc_withheld_ticket = -1;

// Bounded wait that also gives up as soon as another role has aborted.  The
// first test is inline; the sleeping loop is one shared out-of-line copy.
__device__ __noinline__ bool bwait_slow(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    const uint64_t limit = g_tc_wait_ns;
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
            else if (now - t0 > limit) {
                *abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    return mbar_test_wait(bar, parity) || bwait_slow(bar, parity, abort);
}

// Bounded wait used only while draining (ignores the abort flag).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer(), limit = g_tc_wait_ns;
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > limit)
            return;
}

// D (+)= [V | e]^T phi(K) over one 128-token stage: V at vaddr and phi(K) at
// kaddr (MN-major, 128-byte swizzle), e the constant block at `ones`.  The
// second 64 rows of A are read at start + LBO; every K step advances the start
// by 2 KiB, so LBO shrinks by the same amount to keep hitting the one block.
// Executed by a whole warp; the lane with `issue` set issues.
__device__ __forceinline__ void state_mma(uint32_t d, uint32_t vaddr, uint32_t kaddr,
                                          uint32_t ones, bool acc, uint32_t issue)
{
    const uint32_t id = idesc_bf16_f32(128, 64, true, true);
    const uint64_t a0 = sdesc_sw128(vaddr, ones - vaddr, 1024);
    const uint64_t b0 = sdesc_sw128(kaddr, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t step = static_cast<uint64_t>(kk * 128);
        mma_bf16_ss_w(d, a0 + step - (step << 16), b0 + step, id, acc || kk > 0, issue);
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
// and phase C of local segment j-kLag (run by output group (j-kLag) & 1, which
// may still be on it in the next round); the round between a segment's phases
// hides its look-back.
constexpr int kLag = 1;
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

// Every role but the producer walks the same rounds: it learns the A ticket
// of round j from the producer's ring (seg_full) and carries the C ticket kLag
// rounds behind.  A thread group waits through its leader on named barrier
// `barid` (a single thread passes barid < 0).  Returns false when the CTA has
// no more work (or aborted).
struct RoundWalker {
    int h1 = -1, h2 = -1;
    bool doneA = false;
    __device__ __forceinline__ bool next(const TcParams& p, Misc* m, Round& r, int j, bool lead,
                                         int barid, int count, volatile int* abort)
    {
        int tA = -1;
        if (!doneA) {
            int okw = !lead || bwait(&m->seg_full[j % NS], (j / NS) & 1, abort);
            if (barid >= 0)
                okw = group_ok(okw, barid, count);
            if (!okw)
                return false;
            const int t = m->seg_ticket[j % NS];
            if (t < p.total)
                tA = t;
            else
                doneA = true;
        }
        round_setup(p, r, j, tA, kLag == 1 ? h1 : h2);
        h2 = h1;
        h1 = tA;
        return !(r.nA == 0 && r.nC == 0 && (kLag == 1 || h2 < 0));
    }
};

__global__ void __launch_bounds__(kThreads, 1) k_fwd_tc64(const __grid_constant__ TcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Misc* m = reinterpret_cast<Misc*>(sm + OFF_MISC);
    volatile int* abort = &m->abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool norm = p.fm != LA_FM_NONE;
    const uint64_t wait_ns = g_tc_wait_ns;
    const int withheld = g_tc_withheld_ticket;
    const bool elu = p.fm == LA_FM_ELU1;
    const unsigned full = 0xffffffffu;

    if (tid == 0) {
        uint64_t* bars = reinterpret_cast<uint64_t*>(m);
        const int nbars = static_cast<int>((reinterpret_cast<uint64_t*>(&m->drain[4]) - bars) + 1);
        for (int i = 0; i < nbars; ++i)
            mbar_init(&bars[i], 1);
        // a phase-A stage is free once its MMA is done and its phi(K) tile
        // has been copied out
        for (int i = 0; i < NA; ++i)
            mbar_init(&m->a_empty[i], 2);
        m->abort = 0;
        m->trace_done = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.mq);
        tma_prefetch_desc(&p.mk);
        tma_prefetch_desc(&p.mv);
        tma_prefetch_desc(&p.mphi);
    }
    // the e block of [V | e]: element 0 of each of its 16 rows is 1, the rest 0
    // (128-byte swizzle: 16-byte chunk 0 of row r sits at chunk r & 7)
    if (tid < 128) {
        const int r = tid >> 3, c = tid & 7;
        uint4 w = make_uint4(0, 0, 0, 0);
        if (c == (r & 7))
            w.x = 0x3F80u;  // bf16 1.0 in the low half
        *reinterpret_cast<uint4*>(sm + OFF_ONES + r * 128 + c * 16) = w;
    }
    // rows 65..79 of both groups' [S_prev^T; z_prev] operands (hi and lo)
    // stay zero
    for (int i = tid; i < 4 * 15 * 8; i += kThreads) {
        const int t = i / 120, rr = 65 + (i % 120) / 8, c = i % 8;
        *reinterpret_cast<uint4*>(sm + OFF_CW + (t >> 1) * kCWBytes + CW_S + (t & 1) * kSBytes +
                                  rr * 128 + c * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(&m->tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = m->tmem;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ones = smem_addr(sm + OFF_ONES);
    // phi(K) scratch tile of local segment jj, chunk k
    auto phi_index = [&](int jj, int k) {
        return (static_cast<int>(blockIdx.x) * NPH + jj % NPH) * p.L + k;
    };
    // operand image of S_in of local segment jj
    auto sin_img = [&](int jj) {
        return p.sin_img + (static_cast<size_t>(blockIdx.x) * NSIN + jj % NSIN) * kImgBytes;
    };

    if (warp == 0) {
        // ------------------------------------------ producer (one thread) --
        // Three load streams, each advanced as soon as its next step is free:
        // the tickets with the phase-A K,V stages, and the phase-C loads of
        // each output warpgroup.  Local segment jc goes to output group jc & 1,
        // whose chunk loads are: Q once its previous scores and phi(Q)
        // products are done; phi(K) (with the segment's S_in image for its
        // first chunk) and V once its previous chunk's last MMA is done and
        // the segment's phi(K) tiles and S_in are out.
        if (lane == 0) {
            const uint64_t keep = policy_evict_last();
            const uint64_t stream = policy_evict_first();
            int a_last[NA];
            for (int i = 0; i < NA; ++i)
                a_last[i] = -1;
            int ja = 0, ka = 0, ai = 0, nt = 0;  // nt: tickets published
            bool a_seg = false, a_done = false;
            Seg ga{};
            struct CStream {
                int jc = 0, k = 0, u = 0, step = 0;
                int q_last = -1, k_last = -1, v_last = -1;
                bool seg = false, done = false;
                Seg g{};
            } cs[2];
            cs[1].jc = 1;
            uint64_t idle_since = 0;
            while (!(a_done && cs[0].done && cs[1].done)) {
                bool prog = false;
                if (!a_done) {
                    if (!a_seg) {
                        const int ss = ja % NS;
                        if (ja < NS || mbar_test_wait(&m->seg_empty[ss], ((ja / NS) & 1) ^ 1)) {
                            const int t = static_cast<int>(atomicAdd(p.counter, 1u));
                            m->seg_ticket[ss] = t;
                            mbar_arrive(&m->seg_full[ss]);
                            ++nt;
                            prog = true;
                            if (t >= p.total) {
                                a_done = true;
                            } else {
                                ga = seg_of(p, t);
                                ka = 0;
                                a_seg = true;
                            }
                        }
                    } else {
                        const int s = ai % NA;
                        if (ai < NA || mbar_test_wait(&m->a_empty[s], ((ai / NA) & 1) ^ 1)) {
                            mbar_arrive_expect_tx(&m->a_full[s], 2 * kC * kD * 2);
                            unsigned char* st = sm + OFF_A + s * 32768;
                            tma_load_3d(st + 16384, &p.mk, 0, (ga.c0 + ka) * kC, ga.s, &m->a_full[s],
                                        stream);
                            tma_load_3d(st, &p.mv, 0, (ga.c0 + ka) * kC, ga.s, &m->a_full[s], keep);
                            a_last[s] = ai / NA;
                            ++ai;
                            prog = true;
                            if (++ka == ga.n) {
                                a_seg = false;
                                ++ja;
                            }
                        }
                    }
                }
#pragma unroll
                for (int wg = 0; wg < 2; ++wg) {
                    CStream& c = cs[wg];
                    if (c.done)
                        continue;
                    if (!c.seg) {  // this group's next segment, once its ticket is out
                        if (c.jc >= nt) {
                            if (a_done)  // past the last ticket
                                c.done = true;
                            continue;
                        }
                        const int t = m->seg_ticket[c.jc % NS];
                        prog = true;
                        if (t >= p.total) {
                            c.done = true;
                            continue;
                        }
                        c.g = seg_of(p, t);
                        c.k = 0;
                        c.seg = true;
                    }
                    unsigned char* cw = sm + OFF_CW + wg * kCWBytes;
                    const int row = (c.g.c0 + c.k) * kC;
                    if (c.step == 0 &&
                        (c.u == 0 || mbar_test_wait(&m->qs_free[wg], (c.u - 1) & 1))) {
                        mbar_arrive_expect_tx(&m->q_full[wg], kC * kD * 2);
                        tma_load_3d(cw + CW_Q, &p.mq, 0, row, c.g.s, &m->q_full[wg], stream);
                        c.q_last = c.u;
                        c.step = 1;
                        prog = true;
                    }
                    if (c.step == 1 &&
                        (c.u == 0 || mbar_test_wait(&m->ds_done[wg], (c.u - 1) & 1)) &&
                        (c.k > 0 ||
                         (mbar_test_wait(&m->phik_stored[c.jc % NPH], (c.jc / NPH) & 1) &&
                          mbar_test_wait(&m->sin_ready[c.jc % NSIN], (c.jc / NSIN) & 1)))) {
                        mbar_arrive_expect_tx(&m->k_full[wg], kC * kD * 2 + (c.k ? 0 : kImgBytes));
                        tma_load_3d(cw + CW_K, &p.mphi, 0, 0, phi_index(c.jc, c.k), &m->k_full[wg],
                                    stream);
                        if (c.k == 0) {  // the segment's S_in starts the running state
                            const unsigned char* img = sin_img(c.jc);
                            bulk_load(cw + CW_S, img, kImgPart, &m->k_full[wg], stream);
                            bulk_load(cw + CW_S + kSBytes, img + kImgPart, kImgPart,
                                      &m->k_full[wg], stream);
                        }
                        mbar_arrive_expect_tx(&m->v_full[wg], kC * kD * 2);
                        tma_load_3d(cw + CW_V, &p.mv, 0, row, c.g.s, &m->v_full[wg], stream);
                        c.k_last = c.v_last = c.u;
                        c.step = 0;
                        ++c.u;
                        prog = true;
                        if (++c.k == c.g.n) {
                            c.seg = false;
                            c.jc += 2;
                        }
                    }
                }
                if (prog) {
                    idle_since = 0;
                } else {
                    if (*abort)
                        break;
                    const uint64_t now = globaltimer();
                    if (!idle_since) {
                        idle_since = now;
                    } else if (now - idle_since > wait_ns) {
                        set_status(p.status, LA_ERR_TIMEOUT);
                        *abort = 1;
                        break;
                    }
                    __nanosleep(32);
                }
            }
            if (*abort) {  // let every load this thread issued land before exit
                for (int i = 0; i < NA; ++i)
                    if (a_last[i] >= 0)
                        drain_wait(&m->a_full[i], a_last[i] & 1);
                for (int wg = 0; wg < 2; ++wg) {
                    if (cs[wg].q_last >= 0)
                        drain_wait(&m->q_full[wg], cs[wg].q_last & 1);
                    if (cs[wg].k_last >= 0)
                        drain_wait(&m->k_full[wg], cs[wg].k_last & 1);
                    if (cs[wg].v_last >= 0)
                        drain_wait(&m->v_full[wg], cs[wg].v_last & 1);
                }
            }
        }
    } else if (warp < 4) {
        // ------------------------------------ look-back (warps 1-3) --------
        // For each segment whose aggregate phase A has published: what the
        // predecessors have published, the nearest exclusive prefix with that
        // segment's aggregate and every aggregate after it, summed farthest
        // first, gives S_in of this segment bitwise equal to adding the
        // aggregates one by one from the start of the sequence.  S_in goes to
        // the output warpgroups and is published as this segment's exclusive
        // prefix.
        constexpr int kLB = 96, barLB = 4;
        const int tl = tid - 32;
        const bool lead = tl == 0;
        bool ok = true;
        RoundWalker w;
        Round r;
        for (int j = 0; ok && w.next(p, m, r, j, lead, barLB, kLB, abort); ++j) {
            if (!r.nA)
                continue;
            if (!group_ok(!lead || (bwait(&m->agg_ready[j % NSIN], (j / NSIN) & 1, abort) &&
                                    (j < NSIN || bwait(&m->sin_free[j % NSIN],
                                                       ((j / NSIN) & 1) ^ 1, abort))),
                          barLB, kLB)) {
                ok = false;
                break;
            }
            const int t = r.tA, gi = t / p.BH, my = gi % p.R;
            unsigned* flag_base = p.flags + static_cast<size_t>(r.gA.s) * p.R;
            float* slot_base = p.slots + static_cast<size_t>(r.gA.s) * p.R * kSlotFloats;
            if (lead)
                TC_TRACE(j, 5);
            if (warp == 1) {
                // Lane l watches segment base - l.  With a wrapping ring only
                // R-1 slots behind this segment are distinct from its own; a
                // slot holding another epoch reads as not ready.  List entries
                // are slot << 1 | part (0: aggregate, 1: exclusive prefix),
                // nearest first.
                const int W = p.R >= p.nseg ? 32 : min(32, p.R - 1);
                const unsigned active = W >= 32 ? 0xffffffffu : ((1u << W) - 1u);
                int n = 0, base = gi - 1;
                uint64_t start = 0;
                while (base >= 0) {
                    const int pg = base - lane;
                    bool ready = true, excl = true;
                    if (lane >= W) {
                        ready = excl = false;
                    } else if (pg >= 0) {
                        const unsigned f = ld_acquire(flag_base + pg % p.R);
                        ready = (f >> 2) == static_cast<unsigned>(pg + 1) && (f & 3u) != 0u;
                        excl = ready && (f & 3u) == 2u;
                    }
                    const unsigned mi = __ballot_sync(full, excl) & active;
                    const unsigned mr = __ballot_sync(full, ready) & active;
                    if (mi) {
                        const int ls = __ffs(mi) - 1;
                        const unsigned need = ls == 0 ? 0u : ((1u << ls) - 1u);
                        if ((mr & need) == need) {
                            const int tail = base - ls >= 0 ? 2 : 0;
                            if (n + ls + tail > kMaxList) {
                                n = -2;
                                break;
                            }
                            if (lane < ls)
                                m->list[n + lane] = (pg % p.R) << 1;
                            if (lane == ls && tail) {
                                m->list[n + ls] = (pg % p.R) << 1;
                                m->list[n + ls + 1] = ((pg % p.R) << 1) | 1;
                            }
                            n += ls + tail;
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
                    if (__any_sync(full, now - start > wait_ns || *abort)) {
                        n = -1;
                        break;
                    }
                    __nanosleep(64);
                }
                if (lane == 0) {
                    m->nlist = n;
                    if (n < 0) {
                        set_status(p.status, n == -1 ? LA_ERR_TIMEOUT : LA_ERR_DEVICE_CHECK);
                        *abort = 1;
                    }
                }
            }
            named_bar(barLB, kLB);
            const int n = m->nlist;
            if (n < 0) {
                ok = false;
                break;
            }
            if (lead) {
                TC_TRACE(j, 11);
#ifdef LA_TC_TRACE
                if (g_tc_trace && j < 64)
                    g_tc_trace[(static_cast<size_t>(blockIdx.x) * 64 + j) * 32 + 21] = n;
#endif
            }
            // thread tl owns float4 words tl + 96 v of the state
            constexpr int NV = (kStateFloats / 4 + kLB - 1) / kLB;  // 11
            float4 acc[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v)
                acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int e = n - 1; e >= 0; --e) {
                const int ent = m->list[e];
                const float4* src = reinterpret_cast<const float4*>(
                    slot_base + static_cast<size_t>(ent >> 1) * kSlotFloats +
                    ((ent & 1) ? kStateFloats : 0));
                float4 x[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    if (tl + kLB * v < kStateFloats / 4)
                        x[v] = __ldcg(src + tl + kLB * v);
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    if (tl + kLB * v < kStateFloats / 4)
                        acc[v].x += x[v].x, acc[v].y += x[v].y, acc[v].z += x[v].z,
                            acc[v].w += x[v].w;
            }
            // S_in as the operand image the output groups read: bf16 hi and lo
            // parts of rows 0..64 in the 128-byte swizzled slot layout
            unsigned char* img = sin_img(j);
            float4* exc = reinterpret_cast<float4*>(slot_base + static_cast<size_t>(my) * kSlotFloats +
                                                    kStateFloats);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int f = tl + kLB * v;
                if (f < kStateFloats / 4) {
                    __stcg(exc + f, acc[v]);
                    const int row = f >> 4, q = f & 15;
                    uint32_t h0, l0, h1, l1;
                    split2(acc[v].x, acc[v].y, h0, l0);
                    split2(acc[v].z, acc[v].w, h1, l1);
                    const uint32_t off = sw128_off(row, q >> 1) + (q & 1) * 8;
                    __stcg(reinterpret_cast<uint2*>(img + off), make_uint2(h0, h1));
                    __stcg(reinterpret_cast<uint2*>(img + kImgPart + off), make_uint2(l0, l1));
                }
            }
            if (lead)
                TC_TRACE(j, 22);
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __threadfence();
            named_bar(barLB, kLB);
            if (lead) {
                TC_TRACE(j, 23);
                if (t != withheld)
                    st_release(flag_base + my, (static_cast<unsigned>(gi + 1) << 2) | 2u);
                mbar_arrive(&m->sin_ready[j % NSIN]);
                TC_TRACE(j, 12);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // -------------------------- phase A (warpgroup of warps 4-7) --------
        // phi(K) in place, copied to the scratch ring; the segment's running
        // [dS^T; dz] on the tensor cores (warp 4 issues), read out at the end
        // of the segment as its aggregate, which is published for the
        // look-back warps and the other segments.
        const int tb = tid - 128, wb = warp - 4;
        const bool lead = tb == 0;
        const uint32_t issue = wb == 0 ? elect_one() : 0u;
        const uint32_t a0 = smem_addr(sm + OFF_A);
        const uint64_t keep = policy_evict_last();
        int ai = 0;
        bool ok = true, issued = false;
        // [dS^T; dz] so far (tensor-memory lanes 0..64) copied to dst
        auto readout = [&](int x, float* dst) -> bool {
            if (!group_ok(!lead || bwait(&m->dseg_done, x & 1, abort), 1, 128))
                return false;
            tc_fence_after();
            if (wb < 3) {
                uint32_t rr[4][16];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tmem_ld16(tm + TM_DSEG + lane_off + 16 * q, rr[q]);
                tmem_ld_wait();
                if (tb <= kD) {
                    float4* d4 = reinterpret_cast<float4*>(dst + tb * kD);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            __stcg(d4 + 4 * q + u, make_float4(__uint_as_float(rr[q][4 * u]),
                                                               __uint_as_float(rr[q][4 * u + 1]),
                                                               __uint_as_float(rr[q][4 * u + 2]),
                                                               __uint_as_float(rr[q][4 * u + 3])));
                }
            }
            tc_fence_before();
            named_bar(1, 128);
            return true;
        };
        RoundWalker w;
        Round r;
        for (int j = 0; ok && w.next(p, m, r, j, lead, 1, 128, abort); ++j) {
            for (int k = 0; k < r.nA; ++k, ++ai) {
                const int s = ai % NA;
                if (!group_ok(!lead || bwait(&m->a_full[s], (ai / NA) & 1, abort), 1, 128)) {
                    ok = false;
                    break;
                }
                unsigned char* ktile = sm + OFF_A + s * 32768 + 16384;
                if (lead)
                    TC_TRACE(ai, 9);
                phi_tile(ktile, tb, chunk_valid(p, r.gA.c0 + k), elu);
                fence_proxy_async_smem();
                named_bar(1, 128);
                if (lead) {  // phi(K) is kept for phase C in the scratch
                    tma_store_3d(&p.mphi, ktile, 0, 0, phi_index(j, k), keep);
                    bulk_commit();
                    TC_TRACE(ai, 25);
                }
                if (wb == 0) {
                    tc_fence_after();
                    state_mma(tm + TM_DSEG, a0 + s * 32768, a0 + s * 32768 + 16384, ones, k > 0,
                              issue);
                    mma_commit_w(&m->dseg_done, issue);
                    mma_commit_w(&m->a_empty[s], issue);
                    issued = true;
                    if (lead)
                        TC_TRACE(ai, 10);
                }
                if (lead) {  // the stage is free once its copy has read it
                    bulk_wait_read<0>();
                    mbar_arrive(&m->a_empty[s]);
                }
                if (k == r.nA - 1) {  // segment aggregate complete: publish it
                    if (lead)
                        TC_TRACE(j, 15);
                    const int gi = r.tA / p.BH;
                    float* agg =
                        p.slots + (static_cast<size_t>(r.gA.s) * p.R + gi % p.R) * kSlotFloats;
                    if (!(ok = readout(ai, agg)))
                        break;
                    if (lead) {
                        __threadfence();
                        if (r.tA != withheld)
                            st_release(p.flags + static_cast<size_t>(r.gA.s) * p.R + gi % p.R,
                                       (static_cast<unsigned>(gi + 1) << 2) | 1u);
                        // the segment's phi(K) tiles are all in the scratch
                        bulk_wait<0>();
                        mbar_arrive(&m->phik_stored[j % NPH]);
                        mbar_arrive(&m->agg_ready[j % NSIN]);
                        TC_TRACE(j, 24);
                    }
                }
            }
        }
        if (lead)  // no copy may still read a stage
            bulk_wait<0>();
        if (issued && *abort) {
            mma_commit_w(&m->drain[0], issue);
            drain_wait(&m->drain[0], 0);
        }
    } else if (warp >= 8) {
        // ------------------- phase C (warpgroups of warps 8-11 and 12-15) ---
        // Warpgroup wg takes the segments jc with jc & 1 == wg and runs their
        // chunks in order through: phi(Q), scores, P, [num | den], epilogue.
        // Its operand slot holds [S_prev^T; z_prev] as bf16 hi/lo: S_in of
        // the segment at first, then after each chunk but the last the chunk's
        // [dS^T; dz] (computed on the tensor cores) is added in place.  Its
        // first warp issues the MMAs.
        const int wg = (warp - 8) >> 2;
        const int tc = tid - 256 - 128 * wg;   // row of the chunk = tensor-memory lane
        const int wq = tc >> 5;                // 32-row block
        const bool lead = tc == 0;
        const int barid = 2 + wg;
        const uint32_t issue = wq == 0 ? elect_one() : 0u;
        const uint32_t issue3 = wq == 3 ? elect_one() : 0u;
        bool issued3 = false;
        unsigned char* cw = sm + OFF_CW + wg * kCWBytes;
        const uint32_t cwa = smem_addr(cw);
        const uint32_t id_sc = idesc_bf16_f32(128, 128, false, false);
        const uint32_t id_pv = idesc_bf16_f32(128, kON, false, true);
        const uint32_t id_in = idesc_bf16_f32(128, kON, false, false);
        const uint32_t tp = tm + TM_P + 128 * wg, to = tm + TM_O + kON * wg;
        int u = 0;
        bool ok = true, issued = false;
        RoundWalker w;
        Round r;
        for (int j = 0; ok && w.next(p, m, r, j, lead, barid, 128, abort); ++j) {
            const int jc = j - kLag;
            if (!r.nC || (jc & 1) != wg)
                continue;
            for (int k = 0; k < r.nC && ok; ++k, ++u) {
                const bool last = k == r.nC - 1;
                // phi(Q) of the chunk in place, each warp as soon as Q is in
                const bool okq = __all_sync(full, bwait(&m->q_full[wg], u & 1, abort));
                if (okq) {
                    phi_tile(cw + CW_Q, tc, chunk_valid(p, r.gC.c0 + k), elu);
                    fence_proxy_async_smem();
                }
                if (!group_ok(okq, barid, 128)) {
                    ok = false;
                    break;
                }
                // scores, then phi(Q) [S_prev^T; z_prev] (hi, lo) starts the
                // output accumulator while P is prepared
                if (wq == 0 && __all_sync(full, bwait(&m->k_full[wg], u & 1, abort))) {
                    tc_fence_after();
                    const uint64_t dq = sdesc_sw128(cwa + CW_Q, 16, 1024);
                    const uint64_t dk = sdesc_sw128(cwa + CW_K, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss_w(tp, dq + 2 * kk, dk + 2 * kk, id_sc, kk > 0, issue);
                    mma_commit_w(&m->s_done[wg], issue);
                    const uint64_t ds = sdesc_sw128(cwa + CW_S, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss_w(to, dq + 2 * kk, ds + 2 * kk, id_in, kk > 0, issue);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ss_w(to, dq + 2 * kk, ds + (kSBytes >> 4) + 2 * kk, id_in, 1,
                                      issue);
                    mma_commit_w(&m->qs_free[wg], issue);  // the Q slot may refill
                    issued = true;
                }
                // each warp starts its part of P as soon as the scores are in
                // (the issuing warp may still be issuing); verdicts merge below
                const bool okw = __all_sync(full, bwait(&m->s_done[wg], u & 1, abort));
                tc_fence_after();
                // P = tril(scores) as bf16 hi/lo, in place: keys 32q..32q+31 of
                // row tc move to columns 32q..32q+15 (hi) and 32q+16..32q+31 (lo).
                // Blocks left of the diagonal are kept whole, the diagonal block
                // is masked, blocks right of it become zero.
                {
                    const uint32_t pb = tp + lane_off;
#pragma unroll 1
                    for (int q = 0; q <= (okw ? wq : -1); ++q) {
                        uint32_t v0[16], v1[16], hi[16], lo[16];
                        tmem_ld16(pb + 32 * q, v0);
                        tmem_ld16(pb + 32 * q + 16, v1);
                        tmem_ld_wait();
                        if (q < wq) {
#pragma unroll
                            for (int mm = 0; mm < 8; ++mm) {
                                split2(__uint_as_float(v0[2 * mm]), __uint_as_float(v0[2 * mm + 1]),
                                       hi[mm], lo[mm]);
                                split2(__uint_as_float(v1[2 * mm]), __uint_as_float(v1[2 * mm + 1]),
                                       hi[8 + mm], lo[8 + mm]);
                            }
                        } else {
#pragma unroll
                            for (int mm = 0; mm < 8; ++mm) {
                                split2(2 * mm <= lane ? __uint_as_float(v0[2 * mm]) : 0.f,
                                       2 * mm + 1 <= lane ? __uint_as_float(v0[2 * mm + 1]) : 0.f,
                                       hi[mm], lo[mm]);
                                split2(16 + 2 * mm <= lane ? __uint_as_float(v1[2 * mm]) : 0.f,
                                       17 + 2 * mm <= lane ? __uint_as_float(v1[2 * mm + 1]) : 0.f,
                                       hi[8 + mm], lo[8 + mm]);
                            }
                        }
                        tmem_st16(pb + 32 * q, hi);
                        tmem_st16(pb + 32 * q + 16, lo);
                    }
                    uint32_t zz[16];
#pragma unroll
                    for (int mm = 0; mm < 16; ++mm)
                        zz[mm] = 0u;
#pragma unroll 1
                    for (int q = wq + 1; q < 4; ++q) {
                        tmem_st16(pb + 32 * q, zz);
                        tmem_st16(pb + 32 * q + 16, zz);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                if (!group_ok(okw, barid, 128)) {
                    ok = false;
                    break;
                }
                // [num | den] += P [V | e] (P hi/lo pairs), once V is in
                if (wq == 0 && __all_sync(full, bwait(&m->v_full[wg], u & 1, abort))) {
                    tc_fence_after();
                    const uint32_t vs = cwa + CW_V;
                    const uint64_t bv = sdesc_sw128(vs, ones - vs, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t step = static_cast<uint64_t>(kk * 128);
                        mma_bf16_ts_w(to, tp + 32 * (kk >> 1) + 8 * (kk & 1),
                                      bv + step - (step << 16), id_pv, 1, issue);
                    }
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t step = static_cast<uint64_t>(kk * 128);
                        mma_bf16_ts_w(to, tp + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                                      bv + step - (step << 16), id_pv, 1, issue);
                    }
                    mma_commit_w(&m->o_done[wg], issue);
                }
                if (!group_ok(!lead || bwait(&m->o_done[wg], u & 1, abort), barid, 128)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the chunk's [dS^T; dz] = [V | e]^T phi(K) into the score
                // columns (free now) while the epilogue runs; after a segment's
                // last chunk only the slots are handed back
                if (wq == 3) {  // the warp with no state rows to update issues it
                    if (!last)
                        state_mma(tp, cwa + CW_V, cwa + CW_K, ones, false, issue3);
                    mma_commit_w(&m->ds_done[wg], issue3);
                    issued3 = true;
                }
                // epilogue: o = num / den straight from registers.  A 16x256b
                // tensor-memory load gives each quad of threads 8 consecutive
                // columns of one row, so every store fills whole 32-byte sectors;
                // each row's 1/den comes from the thread that owns the row.
                {
                    const float dn = __uint_as_float(tmem_ld1(to + lane_off + kD));
                    tmem_ld_wait();
                    const float inv_row = norm ? 1.0f / fmaxf(dn, FLT_MIN) : 1.0f;
                    const int valid = chunk_valid(p, r.gC.c0 + k);
                    float* obase = p.out + (static_cast<size_t>(r.gC.s) * p.N +
                                            static_cast<size_t>(r.gC.c0 + k) * kC) *
                                               kD;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t rr[32];
                        tmem_ld16x256b_x8(to + lane_off + (static_cast<uint32_t>(16 * h) << 16), rr);
                        tmem_ld_wait();
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int rw = 16 * h + 8 * hr + (lane >> 2);  // row within the warp
                            const float inv = __shfl_sync(full, inv_row, rw);
                            const int row = 32 * wq + rw;
                            // thread q of a quad holds columns 8i + 2q, 8i + 2q + 1;
                            // neighbours swap one pair so the even thread owns
                            // columns 8i + 2q .. 8i + 2q + 3 and the odd one those
                            // of group i + 1, and every store is 16 bytes
                            const bool odd = lane & 1;
                            float* orow = obase + row * kD + 2 * ((lane & 3) & ~1);
#pragma unroll
                            for (int i = 0; i < 8; i += 2) {
                                const float2 g0 = mul2(
                                    make_float2(__uint_as_float(rr[4 * i + 2 * hr]),
                                                __uint_as_float(rr[4 * i + 2 * hr + 1])),
                                    make_float2(inv, inv));
                                const float2 g1 = mul2(
                                    make_float2(__uint_as_float(rr[4 * (i + 1) + 2 * hr]),
                                                __uint_as_float(rr[4 * (i + 1) + 2 * hr + 1])),
                                    make_float2(inv, inv));
                                const float2 give = odd ? g0 : g1;
                                const float2 got = make_float2(__shfl_xor_sync(full, give.x, 1),
                                                               __shfl_xor_sync(full, give.y, 1));
                                if (row < valid) {
                                    const float4 v4 = odd ? make_float4(got.x, got.y, g1.x, g1.y)
                                                          : make_float4(g0.x, g0.y, got.x, got.y);
                                    __stcs(reinterpret_cast<float4*>(orow + 8 * (i + (odd ? 1 : 0))),
                                           v4);
                                }
                            }
                        }
                    }
                }
                bool okd = true;
                if (!last) {
                    // S_prev += [dS^T; dz] in the operand slot: row tc (0..64) of
                    // the hi and lo parts, added in fp32 and split again
                    // each warp with state rows starts once the chunk's update is in
                    okd = wq == 3 || __all_sync(full, bwait(&m->ds_done[wg], u & 1, abort));
                    tc_fence_after();
                    if (wq < 3 && okd) {
                        unsigned char* shi = cw + CW_S;
                        unsigned char* slo = shi + kSBytes;
#pragma unroll 1
                        for (int q = 0; q < 4; ++q) {
                            uint32_t dd[16];
                            tmem_ld16(tp + lane_off + 16 * q, dd);
                            tmem_ld_wait();
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                if (tc > kD)
                                    break;
                                const int cc = 2 * q + hh;
                                const uint32_t off = sw128_off(tc, cc);
                                const uint4 h = *reinterpret_cast<const uint4*>(shi + off);
                                const uint4 l = *reinterpret_cast<const uint4*>(slo + off);
                                const uint32_t* d8 = &dd[8 * hh];
                                const uint32_t hv[4] = {h.x, h.y, h.z, h.w};
                                const uint32_t lv[4] = {l.x, l.y, l.z, l.w};
                                uint32_t nh[4], nl[4];
#pragma unroll
                                for (int t2 = 0; t2 < 4; ++t2) {
                                    const float a = bf_lo(hv[t2]) + bf_lo(lv[t2]) +
                                                    __uint_as_float(d8[2 * t2]);
                                    const float b = bf_hi(hv[t2]) + bf_hi(lv[t2]) +
                                                    __uint_as_float(d8[2 * t2 + 1]);
                                    split2(a, b, nh[t2], nl[t2]);
                                }
                                *reinterpret_cast<uint4*>(shi + off) =
                                    make_uint4(nh[0], nh[1], nh[2], nh[3]);
                                *reinterpret_cast<uint4*>(slo + off) =
                                    make_uint4(nl[0], nl[1], nl[2], nl[3]);
                            }
                        }
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                if (!group_ok(okd, barid, 128)) {
                    ok = false;
                    break;
                }
                // the chunk's phi(K) tile has had its last reader
                l2_discard(static_cast<unsigned char*>(p.phi_scratch) +
                           static_cast<size_t>(phi_index(jc, k)) * (kC * kD * 2) + 128 * tc);
            }
            // done with the segment's S_in and ticket slot
            if (ok && lead) {
                mbar_arrive(&m->sin_free[jc % NSIN]);
                mbar_arrive(&m->seg_empty[jc % NS]);
            }
        }
#ifdef LA_TC_TRACE
        if (lead)
            atomicAdd(const_cast<int*>(&m->trace_done), 1);
#endif
        if (issued && *abort) {
            mma_commit_w(&m->drain[1 + wg], issue);
            drain_wait(&m->drain[1 + wg], 0);
        }
        if (issued3 && *abort) {
            mma_commit_w(&m->drain[3 + wg], issue3);
            drain_wait(&m->drain[3 + wg], 0);
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
    // about eight segments per CTA keeps the tail short; long segments make
    // the look-back rare, and below four chunks a segment's own work (phase
    // A, its slot, the look-back) costs more than the parallelism it buys
    g.L = (int)std::max<int64_t>(kMinL, std::min<int64_t>(kMaxL, chunks / ((int64_t)sms * LA_TC_SEG_DIV)));
    g.L = std::min(g.L, g.nchunk);
    g.nseg = (g.nchunk + g.L - 1) / g.L;
    g.total = (int)(BH * g.nseg);
    int G = sms;
    G = (int)std::min<int64_t>(G, g.total);
    G = (int)std::min<int64_t>(G, BH * kMaxCtasPerSeq);  // bounds the look-back list
    if (G < 1)
        G = 1;
    g.G = G;
    // one slot per segment: a slot is written once per launch, so no reader
    // can ever see it overwritten (a ring sized by the tickets in flight
    // bounds the tickets held, not the span between a slow reader and the
    // newest writer: a later segment can finish its look-back, and a yet
    // later one publish, while an earlier one is still reading)
    g.R = g.nseg;
    g.flags_off = 256;
    g.slots_off = (g.flags_off + sizeof(unsigned) * (size_t)BH * g.R + 255) & ~(size_t)255;
    g.sin_off = g.slots_off + sizeof(float) * (size_t)BH * g.R * kSlotFloats;
    g.sin_off = (g.sin_off + 1023) & ~(size_t)1023;
    g.phi_off = (g.sin_off + (size_t)G * NSIN * kImgBytes + 1023) & ~(size_t)1023;
    g.bytes = g.phi_off + (size_t)G * NPH * g.L * kC * kD * 2;
    return g;
}

}  // namespace

bool tc_forward_eligible(const FwdArgs& a)
{
    // the look-back list bounds this kernel to kMaxCtasPerSeq CTAs per
    // sequence; with fewer sequences than that needs to fill the GPU, the
    // chunked path (which splits each sequence over the whole GPU) serves the
    // call
    const int64_t BH = a.B * a.H;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    return a.dtype == LA_BF16 && a.d == 64 && a.dv == 64 && a.causal == 1 && !a.gamma->has_decay &&
           a.N >= 1 && a.N <= (int64_t)INT32_MAX - kC && BH * kMaxCtasPerSeq >= sms;
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
        !make_map(&p.mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, a.N, BH, 64))
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
    p.sin_img = ws + g.sin_off;
    p.phi_scratch = ws + g.phi_off;
    p.out = static_cast<float*>(a.out);
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

// Test hook of the give-up path (declared in linattn.h).
extern "C" __attribute__((visibility("default"))) la_status la_debug_set_tc_faults(
    uint64_t wait_ns, int withheld_segment)
{
    if (wait_ns == 0)
        return LA_ERR_INVALID_ARG;
    if (cudaMemcpyToSymbol(g_tc_wait_ns, &wait_ns, sizeof wait_ns) != cudaSuccess ||
        cudaMemcpyToSymbol(g_tc_withheld_ticket, &withheld_segment, sizeof(int)) != cudaSuccess)
        return LA_ERR_CUDA;
    return LA_OK;
}

bool tma_map_bf16_3d(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t depth)
{
    return make_map(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, depth, 64);
}

int device_sm_count() { return sm_count(); }

#ifdef LA_TC_TRACE
extern "C" __attribute__((visibility("default"))) int la_debug_set_tc_trace(void* buf)
{
    return (int)cudaMemcpyToSymbol(g_tc_trace, &buf, sizeof(buf));
}
#endif

}  // namespace la
