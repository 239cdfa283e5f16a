// Shared definitions of the MoDA CUDA library (kernels and host dispatch).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace moda {

// log2(e): the slides' Algorithm 1 uses 2^(S-m); folding log2(e) into the score
// scale makes that the natural-exponential softmax of the operation
// (frame "Backup: pseudocode needs implementation-level checks").
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status word codes (mirror moda_status).
constexpr int kStatusConfig = 3;   // a kernel refused its launch configuration (MODA_ERR_CUDA)
constexpr int kStatusTimeout = 4;  // a bounded wait ran out (MODA_ERR_TIMEOUT)

struct Problem {
  int B, H, Hkv, T;
  int Tk;      // key positions per (b, kv head) in k/v (T for a whole sequence)
  int delta;   // key j is visible to query position t iff j <= t + delta (0 for a whole sequence)
  int S;       // depth slots per position in kd/vd memory (0: no depth memory)
  int S_read;  // slots 0 .. S_read-1 of each position are read (S_read <= S; S_read = 0 iff S = 0)
  int d, G;
  float scale;       // score scale (1/sqrt(d) by default)
  float scale_log2;  // scale * log2(e)
};

struct FwdArgs {
  Problem p;
  int* status;  // device status word (bounded-wait timeouts)
  const void *q, *k, *v, *kd, *vd;
  void* o;
  float* lse;  // may be null
};

struct BwdArgs {
  Problem p;
  int* status;
  const void *q, *k, *v, *kd, *vd, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv, *dkd, *dvd;
  float2* stats;    // workspace [B,H,T]: {-lse * log2(e), Delta_t = dout_t . o_t}
  float* dq_accum;  // workspace [B,H,T,d] float32 (tensor-core path)
  // When set (all three), the sequence gradients are added in float32 to these instead
  // of being written to dq/dk/dv: dq_acc [B,H,T,d], dk_acc/dv_acc [B,Hkv,Tk,d].
  float *dq_acc, *dk_acc, *dv_acc;
  void** events;    // optional cudaEvent_t[n_events]: stage k recorded at events[2k] (start), [2k+1] (end)
  int n_events;
};

// Decode step: q [B,H,d] (the newest position of every head), k/v cache [B,Hkv,cap,d]
// holding positions 0 .. T-1, kd/vd [B,Hkv,S,d] (the newest position's depth slots).
struct DecodeArgs {
  Problem p;
  int64_t cap;  // positions allocated per (b, kv head) in the cache (>= T)
  int* status;
  const void *q, *k, *v, *kd, *vd;
  void* o;     // [B,H,d]
  float* lse;  // [B,H], may be null
  float* part; // workspace: per-split partial states
};
struct DecodeSplit {
  int n_seq;    // sequence splits
  int chunk;    // sequence keys per split
  int n_split;  // n_seq (+1 for the depth slots when S > 0)
};

// Depth-KV write path: slot `slot` of kd/vd [B,Hkv,T,S,d] from the attention KV
// (k/v [B,Hkv,T,d]) or from the projection of x [B,T,Dm] by wk/wv [Dm, Hkv*d].
// Merge of a partial forward state (o_part, lse_part) into a running float32 state
// (o_acc, lse_acc), rows = B*H*T rows of d columns; `first`: the running state is set to
// the partial one.  o_out (may be null) receives the merged O in the storage type.
struct MergeArgs {
  int64_t rows;
  int d, first;
  float *o_acc, *lse_acc;
  const void* o_part;
  const float* lse_part;
  void* o_out;
};

struct DepthWriteArgs {
  int B, Hkv, T, S, d, slot, Dm;
  int* status;
  const void *k, *v, *x, *wk, *wv;
  void *kd, *vd;
};

// cuTensorMapEncodeTiled from the driver (looked up once, thread-safe); null when the
// driver does not provide it.
void* tensor_map_encoder();

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current device, once per
// device: the attribute belongs to the kernel's instance on each device, so a process that
// drives several GPUs sets it on each.  `done` is the call site's per-device bit mask
// (devices 0..63; a higher ordinal sets the attribute on every call).  Concurrent callers
// may both set it, which is harmless.
template <typename K>
cudaError_t ensure_dynamic_smem(K kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Records a.events[k] on `s` when the caller asked for it (profiling only).
inline void mark_event(const BwdArgs& a, int k, cudaStream_t s) {
  if (a.events != nullptr && k < a.n_events && a.events[k] != nullptr)
    cudaEventRecord(static_cast<cudaEvent_t>(a.events[k]), s);
}

// Element loads/stores for the two storage types.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Records the first error code in the device status word (never traps).
__device__ __forceinline__ void record_status(int* status, int code) { atomicCAS(status, 0, code); }

// Host-side count of kernels this library has launched (reported by moda_launch_count).
void count_launches(int n);

// Host-side launchers (one per kernel family).  Each returns the launch error.
cudaError_t launch_fwd_simt(const FwdArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_bwd_simt(const BwdArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_bwd_delta(const BwdArgs& a, int dtype, cudaStream_t s);  // Delta = rowsum(dout * o)
cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_fwd_sm103(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_sm103(const BwdArgs& a, cudaStream_t s);
bool fwd_sm103_supported(const Problem& p);
DecodeSplit decode_split(const Problem& p);
bool decode_sm103_supported(const Problem& p);
cudaError_t launch_decode_sm103(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_depth_store_sm103(const DepthWriteArgs& a, cudaStream_t s);
cudaError_t launch_depth_project_sm103(const DepthWriteArgs& a, cudaStream_t s);
bool bwd_sm103_supported(const Problem& p);
cudaError_t launch_merge(const MergeArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_convert(int64_t n, const float* src, void* dst, int dtype, cudaStream_t s);

}  // namespace moda
