// la_internal.cuh -- declarations shared by the CUDA translation units of
// liblinattn.so (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "linattn.h"

namespace la {

constexpr int kMaxGammaHeads = 256;    // per-head decay table passed by value

// Per-head log2(gamma), passed by value in the kernel parameters so that a
// host gamma array needs no device copy.  has_decay = 0 means gamma = 1.
struct GammaTable {
    int has_decay;
    int H;
    float g[kMaxGammaHeads];      // gamma itself (decode multiplies by it)
    float log2g[kMaxGammaHeads];  // log2(gamma) for powers gamma^n
};

// gamma^n for a head, as exp2(n * log2 gamma); exact 1 without decay.
__device__ __forceinline__ float gamma_pow(const GammaTable& g, int head, float n)
{
    return g.has_decay ? exp2f(n * g.log2g[head]) : 1.0f;
}

__device__ __forceinline__ float gamma_one(const GammaTable& g, int head)
{
    return g.has_decay ? g.g[head] : 1.0f;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}

// The feature map in fp32: elu(x)+1 = max(x,0) + exp(min(x,0)), or identity.
__device__ __forceinline__ float phi_f32(float x, int fm)
{
    if (fm != LA_FM_ELU1)
        return x;
    return x > 0.0f ? x + 1.0f : expf(x);
}

__device__ __forceinline__ bool fm_normalised(int fm) { return fm != LA_FM_NONE; }

// Device status codes written by kernels (a subset of la_status).
__device__ __forceinline__ void set_status(int* status, int code)
{
    if (status)
        atomicCAS(status, 0, code);
}

// Count one kernel launch (la_launch_count).
void count_launches(int n);

// ---- workspace layout of the chunked forward ------------------------------
// [BH][nblk][state] fp32 where state = d*dv (S) followed by d (z).
struct ChunkGeom {
    int64_t BH;
    int64_t N;
    int nblk;        // blocks per sequence
    int L;           // tokens per block
    int state_elems; // d*dv + d
};

// ---- launchers (each returns a cudaError_t from the launch) ----------------
struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    float* out;
    int64_t B, H, N;
    int d, dv, causal, fm, dtype;
    GammaTable* gamma;  // host copy; passed by value to kernels
    void* ws;
    size_t ws_bytes;
    float* S_out;       // final state [B,H,d,dv] (else NULL)
    float* z_out;       // final normaliser state [B,H,d] (else NULL)
    const float* S0;    // state before the first token [B,H,d,dv] (else NULL = 0)
    const float* z0;
    int* status;        // device status word
    cudaStream_t stream;
};

size_t simt_forward_workspace(int64_t BH, int64_t N, int d, int dv, int causal);
size_t simt_state_workspace(int64_t BH, int64_t N, int d, int dv);
cudaError_t simt_forward(const FwdArgs& a);
cudaError_t simt_state(const FwdArgs& a);

// tcgen05 / TMA single-pass causal forward (bf16, d = dv = 64, no decay)
bool tc_forward_eligible(const FwdArgs& a);
size_t tc_forward_workspace(int64_t BH, int64_t N);
cudaError_t tc_forward(const FwdArgs& a);

// tcgen05 chunkwise path (bf16, d and dv in {64, 128}): segment aggregates,
// scan, outputs.  Serves forwards (a.out), final states (a.S_out) and initial
// states (a.S0); decay only with the unnormalised map when outputs are wanted.
bool tg_eligible(const FwdArgs& a);
size_t tg_workspace(int64_t BH, int64_t N, int d, int dv, int fm, int causal);
cudaError_t tg_run(const FwdArgs& a);

// A 3D TMA descriptor over a bf16 tensor [depth][rows][cols] (row-major),
// boxes of 128 rows x 64 columns with the 128-byte swizzle.
bool tma_map_bf16_3d(CUtensorMap* m, const void* base, int64_t cols, int64_t rows,
                     int64_t depth);
// Streaming multiprocessors of the current device (0 if unknown).
int device_sm_count();

// per-key-channel decay (GLA): CUDA-core chunked forward
struct GlaArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;  // [B,H,N,d] fp32 in (0, 1]
    float* out;
    int64_t B, H, N;
    int d, dv, fm, dtype;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};
size_t gla_workspace(int64_t BH, int64_t N, int d, int dv);
cudaError_t gla_forward(const GlaArgs& a);

// exclusive prefix of per-part states for a split sequence (la_state_prefix)
int state_prefix_max_parts();
cudaError_t state_prefix(const float* S, const float* z, int nparts, const int64_t* len, int upto,
                         float* S_out, float* z_out, int64_t BH, int H, int d, int dv,
                         const GammaTable& g, cudaStream_t st);

// positive random features (la_favor_features)
bool favor_shape_ok(int d, int r);
cudaError_t favor_features(const void* x, const float* w, void* out, int64_t rows, int d, int r,
                           int in_dtype, int out_dtype, int* status, cudaStream_t st);

struct DecodeArgs {
    float* S;
    float* z;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;  // [B,H,d] per-key-channel decay of this step, or NULL
    float* out;
    int64_t BH, H;
    int d, dv, fm, dtype;
    GammaTable* gamma;
    cudaStream_t stream;
};
cudaError_t decode_step(const DecodeArgs& a);

}  // namespace la
