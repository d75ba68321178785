// la_api.cu -- the C ABI of liblinattn.so: argument checks, dispatch, status.
//
// Every entry point validates its arguments before anything is enqueued and
// never allocates: scratch is the caller's workspace, and the only
// library-owned device object is the per-device status word below, a static
// __device__ variable that exists as soon as the module is loaded.
#include <atomic>
#include <math.h>
#include <mutex>

#include "la_internal.cuh"

namespace la {
__device__ int g_device_status;  // LA_OK, or the first device-side error code

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
int* g_status_ptr[kMaxDevices];

// Device address of the status word for the current device (looked up once).
int* status_ptr()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess)
            return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

bool dim_ok(int x) { return x == 32 || x == 64 || x == 128; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Workspaces hold 128-byte lines that kernels drop from L2 and 1024-byte
// aligned TMA regions laid out from the base, so the base must be 256-aligned.
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

la_status check_sizes(int64_t B, int64_t H, int64_t N, int d, int dv, int fm, int dtype)
{
    if (B < 1 || H < 1 || N < 0 || d < 1 || dv < 1)
        return LA_ERR_INVALID_ARG;
    if (fm != LA_FM_ELU1 && fm != LA_FM_IDENTITY_NORM && fm != LA_FM_NONE)
        return LA_ERR_INVALID_ARG;
    if (dtype != LA_BF16 && dtype != LA_FP32)
        return LA_ERR_INVALID_ARG;
    if (!dim_ok(d) || !dim_ok(dv))
        return LA_ERR_UNSUPPORTED;
    if (B > INT32_MAX / H)
        return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

// Fill the by-value decay table; NULL gamma means no decay.
la_status make_gamma(const float* gamma, int64_t H, GammaTable* t)
{
    t->has_decay = 0;
    t->H = (int)(H < kMaxGammaHeads ? H : kMaxGammaHeads);
    if (!gamma)
        return LA_OK;
    if (H > kMaxGammaHeads)
        return LA_ERR_UNSUPPORTED;
    for (int64_t h = 0; h < H; ++h) {
        const float gm = gamma[h];
        if (!(gm > 0.0f && gm <= 1.0f))
            return LA_ERR_INVALID_ARG;
        t->g[h] = gm;
        t->log2g[h] = (float)log2((double)gm);
    }
    t->has_decay = 1;
    return LA_OK;
}

la_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

}  // namespace
}  // namespace la

using namespace la;

extern "C" {

int la_version(void) { return 100; }  // 0.1.0

const char* la_status_string(la_status s)
{
    switch (s) {
    case LA_OK: return "LA_OK: success";
    case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG: invalid argument (pointer, size, enum or gamma)";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: valid request outside what is implemented";
    case LA_ERR_CUDA: return "LA_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a bounded device-side wait gave up";
    case LA_ERR_DEVICE_CHECK: return "LA_ERR_DEVICE_CHECK: a device-side consistency check failed";
    case LA_ERR_WORKSPACE: return "LA_ERR_WORKSPACE: workspace missing or too small";
    case LA_ERR_TOO_LARGE:
        return "LA_ERR_TOO_LARGE: sizes need more scratch than la_forward_noalloc's fixed array";
    }
    return "unknown la_status";
}

// The kernel paths, in order of preference: the single-pass tcgen05 kernel
// (bf16, d = dv = 64, causal, no decay, no state in or out), the chunked
// tcgen05 path (bf16, d and dv in {64, 128}), the CUDA-core path.
enum Path { PATH_TC = 0, PATH_TG = 1, PATH_SIMT = 2 };

static Path choose_path(const FwdArgs& a)
{
    if (a.out && !a.S0 && !a.S_out && tc_forward_eligible(a))
        return PATH_TC;
    if (tg_eligible(a))
        return PATH_TG;
    return PATH_SIMT;
}

static FwdArgs probe_args(int64_t B, int64_t H, int64_t N, int d, int dv, int causal, int fm,
                          int dtype, GammaTable* g, bool out, bool state)
{
    FwdArgs a{};
    a.B = B, a.H = H, a.N = N, a.d = d, a.dv = dv, a.causal = causal, a.fm = fm;
    a.dtype = dtype, a.gamma = g;
    // placeholders that only mark which results are wanted
    a.out = out ? reinterpret_cast<float*>(uintptr_t(256)) : nullptr;
    a.S_out = state ? reinterpret_cast<float*>(uintptr_t(256)) : nullptr;
    return a;
}

static size_t path_workspace(const FwdArgs& a, Path path)
{
    switch (path) {
    case PATH_TC: return tc_forward_workspace(a.B * a.H, a.N);
    case PATH_TG: return tg_workspace(a.B * a.H, a.N, a.d, a.dv, a.fm, a.causal);
    default:
        return a.out ? simt_forward_workspace(a.B * a.H, a.N, a.d, a.dv, a.causal)
                     : simt_state_workspace(a.B * a.H, a.N, a.d, a.dv);
    }
}

// Workspace that covers every path a call with these sizes may take (the
// feature map and the decay are not known here).
static size_t max_workspace(int64_t B, int64_t H, int64_t N, int d, int dv, int causal,
                            int dtype, bool out, bool state)
{
    size_t n = 0;
    for (int fm = 0; fm < 3; ++fm)
        for (int decay = 0; decay < 2; ++decay) {
            GammaTable g{};
            g.has_decay = decay;
            const FwdArgs a = probe_args(B, H, N, d, dv, causal, fm, dtype, &g, out, state);
            const size_t w = path_workspace(a, choose_path(a));
            n = w > n ? w : n;
        }
    return n;
}

size_t la_forward_workspace_size(int64_t B, int64_t H, int64_t N, int d, int dv, int causal,
                                 int dtype)
{
    if (check_sizes(B, H, N, d, dv, LA_FM_ELU1, dtype) != LA_OK || N == 0)
        return 0;
    // the forward alone, and with states in or out (causal only)
    size_t n = max_workspace(B, H, N, d, dv, causal, dtype, true, false);
    if (causal) {
        const size_t w = max_workspace(B, H, N, d, dv, causal, dtype, true, true);
        n = w > n ? w : n;
    }
    return n;
}

const char* la_forward_path(int64_t B, int64_t H, int64_t N, int d, int dv, int causal,
                            int feature_map, int has_decay, int dtype)
{
    if (check_sizes(B, H, N, d, dv, feature_map, dtype) != LA_OK)
        return "invalid";
    GammaTable g{};
    g.has_decay = has_decay;
    const FwdArgs a = probe_args(B, H, N, d, dv, causal, feature_map, dtype, &g, true, false);
    switch (choose_path(a)) {
    case PATH_TC: return "tcgen05";
    case PATH_TG: return "tcgen05_chunked";
    default: return "simt";
    }
}

size_t la_state_workspace_size(int64_t B, int64_t H, int64_t N, int d, int dv, int dtype)
{
    if (check_sizes(B, H, N, d, dv, LA_FM_ELU1, dtype) != LA_OK || N == 0)
        return 0;
    return max_workspace(B, H, N, d, dv, 1, dtype, false, true);
}

// Runs a validated forward and/or state request on its path.
static la_status run_path(const FwdArgs& a)
{
    const Path path = choose_path(a);
    const size_t need = path_workspace(a, path);
    if (!a.ws || a.ws_bytes < need || !aligned256(a.ws))
        return LA_ERR_WORKSPACE;
    switch (path) {
    case PATH_TC: return from_cuda(tc_forward(a));
    case PATH_TG: return from_cuda(tg_run(a));
    default: return from_cuda(a.out ? simt_forward(a) : simt_state(a));
    }
}

la_status la_forward(const void* q, const void* k, const void* v, float* out, int64_t B,
                     int64_t H, int64_t N, int d, int dv, int causal, int feature_map,
                     const float* gamma, int dtype, void* workspace, size_t workspace_bytes,
                     la_stream_t stream)
{
    la_status st = check_sizes(B, H, N, d, dv, feature_map, dtype);
    if (st != LA_OK)
        return st;
    if (causal != 0 && causal != 1)
        return LA_ERR_INVALID_ARG;
    if (!causal && gamma)
        return LA_ERR_UNSUPPORTED;  // decay is defined only for the causal form
    GammaTable gt;
    if ((st = make_gamma(gamma, H, &gt)) != LA_OK)
        return st;
    if (N == 0)
        return LA_OK;
    if (!q || !k || !v || !out)
        return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return LA_ERR_INVALID_ARG;
    FwdArgs a{};
    a.q = q, a.k = k, a.v = v, a.out = out;
    a.B = B, a.H = H, a.N = N, a.d = d, a.dv = dv;
    a.causal = causal, a.fm = feature_map, a.dtype = dtype;
    a.gamma = &gt;
    a.ws = workspace, a.ws_bytes = workspace_bytes;
    a.status = status_ptr();
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return run_path(a);
}

la_status la_forward_with_state(const void* q, const void* k, const void* v, float* out,
                                const float* S0, const float* z0, float* S_out, float* z_out,
                                int64_t B, int64_t H, int64_t N, int d, int dv, int feature_map,
                                const float* gamma, int dtype, void* workspace,
                                size_t workspace_bytes, la_stream_t stream)
{
    la_status st = check_sizes(B, H, N, d, dv, feature_map, dtype);
    if (st != LA_OK)
        return st;
    GammaTable gt;
    if ((st = make_gamma(gamma, H, &gt)) != LA_OK)
        return st;
    if (!S0 != !z0 || !S_out != !z_out || (!out && !S_out) || (!q != !out))
        return LA_ERR_INVALID_ARG;
    if ((S0 && (!aligned16(S0) || !aligned16(z0))) ||
        (S_out && (!aligned16(S_out) || !aligned16(z_out))))
        return LA_ERR_INVALID_ARG;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) {  // no tokens: the final state is the initial one
        if (!S_out)
            return LA_OK;
        const size_t sb = sizeof(float) * (size_t)(B * H) * d * dv;
        const size_t zb = sizeof(float) * (size_t)(B * H) * d;
        cudaError_t e;
        if (S0) {
            e = S0 == S_out ? cudaSuccess : cudaMemcpyAsync(S_out, S0, sb, cudaMemcpyDeviceToDevice, cs);
            if (e == cudaSuccess && z0 != z_out)
                e = cudaMemcpyAsync(z_out, z0, zb, cudaMemcpyDeviceToDevice, cs);
        } else {
            e = cudaMemsetAsync(S_out, 0, sb, cs);
            if (e == cudaSuccess)
                e = cudaMemsetAsync(z_out, 0, zb, cs);
        }
        return from_cuda(e);
    }
    if (!k || !v || !aligned16(k) || !aligned16(v))
        return LA_ERR_INVALID_ARG;
    if (out && (!aligned16(q) || !aligned16(out)))
        return LA_ERR_INVALID_ARG;
    FwdArgs a{};
    a.q = q, a.k = k, a.v = v, a.out = out;
    a.B = B, a.H = H, a.N = N, a.d = d, a.dv = dv;
    a.causal = 1, a.fm = feature_map, a.dtype = dtype;
    a.gamma = &gt;
    a.ws = workspace, a.ws_bytes = workspace_bytes;
    a.S0 = S0, a.z0 = z0, a.S_out = S_out, a.z_out = z_out;
    a.status = status_ptr();
    a.stream = cs;
    return run_path(a);
}

la_status la_state(const void* k, const void* v, float* S, float* z, int64_t B, int64_t H,
                   int64_t N, int d, int dv, int feature_map, const float* gamma, int dtype,
                   void* workspace, size_t workspace_bytes, la_stream_t stream)
{
    la_status st = check_sizes(B, H, N, d, dv, feature_map, dtype);
    if (st != LA_OK)
        return st;
    GammaTable gt;
    if ((st = make_gamma(gamma, H, &gt)) != LA_OK)
        return st;
    if (!S || !z || !aligned16(S) || !aligned16(z))
        return LA_ERR_INVALID_ARG;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) {
        cudaError_t e = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)(B * H) * d * dv, cs);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(z, 0, sizeof(float) * (size_t)(B * H) * d, cs);
        return from_cuda(e);
    }
    if (!k || !v || !aligned16(k) || !aligned16(v))
        return LA_ERR_INVALID_ARG;
    FwdArgs a{};
    a.k = k, a.v = v;
    a.B = B, a.H = H, a.N = N, a.d = d, a.dv = dv;
    a.causal = 1, a.fm = feature_map, a.dtype = dtype;
    a.gamma = &gt;
    a.ws = workspace, a.ws_bytes = workspace_bytes;
    a.S_out = S, a.z_out = z;
    a.status = status_ptr();
    a.stream = cs;
    return run_path(a);
}

la_status la_decode_step(float* S, float* z, const void* q, const void* k, const void* v,
                         float* out, int64_t B, int64_t H, int d, int dv, int feature_map,
                         const float* gamma, int dtype, la_stream_t stream)
{
    la_status st = check_sizes(B, H, 1, d, dv, feature_map, dtype);
    if (st != LA_OK)
        return st;
    GammaTable gt;
    if ((st = make_gamma(gamma, H, &gt)) != LA_OK)
        return st;
    if (!S || !z || !q || !k || !v || !out)
        return LA_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(z) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(out))
        return LA_ERR_INVALID_ARG;
    DecodeArgs a{};
    a.S = S, a.z = z, a.q = q, a.k = k, a.v = v, a.out = out;
    a.BH = B * H, a.H = H, a.d = d, a.dv = dv, a.fm = feature_map, a.dtype = dtype;
    a.gamma = &gt;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return from_cuda(decode_step(a));
}

size_t la_gla_workspace_size(int64_t B, int64_t H, int64_t N, int d, int dv)
{
    if (check_sizes(B, H, N, d, dv, LA_FM_ELU1, LA_FP32) != LA_OK)
        return 0;
    return gla_workspace(B * H, N, d, dv);
}

la_status la_forward_gla(const void* q, const void* k, const void* v, const float* alpha,
                         float* out, int64_t B, int64_t H, int64_t N, int d, int dv,
                         int feature_map, int dtype, void* workspace, size_t workspace_bytes,
                         la_stream_t stream)
{
    la_status st = check_sizes(B, H, N, d, dv, feature_map, dtype);
    if (st != LA_OK)
        return st;
    if (N == 0)
        return LA_OK;
    if (!q || !k || !v || !alpha || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(alpha) || !aligned16(out))
        return LA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < gla_workspace(B * H, N, d, dv) || !aligned256(workspace))
        return LA_ERR_WORKSPACE;
    GlaArgs a{};
    a.q = q, a.k = k, a.v = v, a.alpha = alpha, a.out = out;
    a.B = B, a.H = H, a.N = N, a.d = d, a.dv = dv, a.fm = feature_map, a.dtype = dtype;
    a.ws = workspace, a.ws_bytes = workspace_bytes;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return from_cuda(gla_forward(a));
}

la_status la_decode_step_gla(float* S, float* z, const void* q, const void* k, const void* v,
                             const float* alpha, float* out, int64_t B, int64_t H, int d, int dv,
                             int feature_map, int dtype, la_stream_t stream)
{
    if (!alpha || !aligned16(alpha))
        return LA_ERR_INVALID_ARG;
    la_status st = check_sizes(B, H, 1, d, dv, feature_map, dtype);
    if (st != LA_OK)
        return st;
    if (!S || !z || !q || !k || !v || !out)
        return LA_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(z) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(out))
        return LA_ERR_INVALID_ARG;
    GammaTable gt;
    make_gamma(nullptr, H, &gt);
    DecodeArgs a{};
    a.S = S, a.z = z, a.q = q, a.k = k, a.v = v, a.alpha = alpha, a.out = out;
    a.BH = B * H, a.H = H, a.d = d, a.dv = dv, a.fm = feature_map, a.dtype = dtype;
    a.gamma = &gt;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return from_cuda(decode_step(a));
}

la_status la_state_prefix(const float* S_parts, const float* z_parts, int nparts,
                          const int64_t* part_len, int upto, float* S_out, float* z_out,
                          int64_t B, int64_t H, int d, int dv, const float* gamma,
                          la_stream_t stream)
{
    la_status st = check_sizes(B, H, 1, d, dv, LA_FM_ELU1, LA_FP32);
    if (st != LA_OK)
        return st;
    GammaTable gt;
    if ((st = make_gamma(gamma, H, &gt)) != LA_OK)
        return st;
    if (nparts < 1 || nparts > state_prefix_max_parts() || upto < 0 || upto > nparts || !part_len)
        return LA_ERR_INVALID_ARG;
    for (int q = 0; q < nparts; ++q)
        if (part_len[q] < 0)
            return LA_ERR_INVALID_ARG;
    if (!S_parts || !z_parts || !S_out || !z_out || !aligned16(S_parts) || !aligned16(z_parts) ||
        !aligned16(S_out) || !aligned16(z_out))
        return LA_ERR_INVALID_ARG;
    return from_cuda(state_prefix(S_parts, z_parts, nparts, part_len, upto, S_out, z_out, B * H,
                                  (int)H, d, dv, gt, reinterpret_cast<cudaStream_t>(stream)));
}

la_status la_favor_features(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                            int in_dtype, int out_dtype, la_stream_t stream)
{
    if (rows < 0 || !favor_shape_ok(d, r))
        return rows < 0 || d < 1 || r < 1 ? LA_ERR_INVALID_ARG : LA_ERR_UNSUPPORTED;
    if ((in_dtype != LA_BF16 && in_dtype != LA_FP32) || (out_dtype != LA_BF16 && out_dtype != LA_FP32))
        return LA_ERR_INVALID_ARG;
    if (rows == 0)
        return LA_OK;
    if (!x || !w || !out || !aligned16(x) || !aligned16(w) || !aligned16(out))
        return LA_ERR_INVALID_ARG;
    return from_cuda(favor_features(x, w, out, rows, d, r, in_dtype, out_dtype, status_ptr(),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

uint64_t la_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

la_status la_get_device_status(la_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess)
        return LA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess)
            return LA_ERR_CUDA;
    }
    return static_cast<la_status>(v);
}

}  // extern "C"
