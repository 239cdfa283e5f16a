// C ABI of the MoDA library (declared in include/moda.h): argument checks,
// kernel selection and launches.  All compute runs in the kernels of this
// directory; nothing here touches tensor data on the host.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moda.h"
#include "moda_common.cuh"

namespace moda {
namespace {
std::atomic<int64_t> g_launches{0};
}
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

void* tensor_map_encoder() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = ptr;
  });
  return fn;
}
}  // namespace moda

namespace {

// Device status word that bounded waits write (MODA_ERR_TIMEOUT) instead of trapping.
__device__ int g_status_word = 0;

constexpr int64_t kMaxElems = int64_t(1) << 40;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t mul_capped(int64_t a, int64_t b) {
  if (a <= 0 || b <= 0) return a * b;
  if (a > kMaxElems / b) return kMaxElems + 1;
  return a * b;
}

// Slots per position in kd/vd memory: slot_capacity when set, else S.
int64_t slots_in_memory(const moda_desc* d) { return d->slot_capacity > 0 ? d->slot_capacity : d->S; }

moda_status check_desc(const moda_desc* d) {
  if (d == nullptr) return MODA_ERR_INVALID_ARG;
  if (d->B < 1 || d->H < 1 || d->Hkv < 1 || d->T < 1 || d->S < 0 || d->d < 1) return MODA_ERR_INVALID_ARG;
  if (d->slot_capacity < 0 || (d->slot_capacity > 0 && d->slot_capacity < d->S)) return MODA_ERR_INVALID_ARG;
  if (d->H % d->Hkv != 0) return MODA_ERR_INVALID_ARG;
  if (!(d->scale <= 0.f || std::isfinite(d->scale))) return MODA_ERR_INVALID_ARG;
  if (d->dtype != MODA_DTYPE_F32 && d->dtype != MODA_DTYPE_BF16) return MODA_ERR_UNSUPPORTED;
  if (d->d != 64 && d->d != 128) return MODA_ERR_UNSUPPORTED;
  const int64_t q = mul_capped(mul_capped(mul_capped(d->B, d->H), d->T), d->d);
  const int64_t kd = mul_capped(mul_capped(mul_capped(mul_capped(d->B, d->Hkv), d->T), slots_in_memory(d)), d->d);
  if (q > kMaxElems || kd > kMaxElems) return MODA_ERR_INVALID_ARG;
  return MODA_OK;
}

moda::Problem problem_of(const moda_desc* d) {
  moda::Problem p;
  p.B = d->B;
  p.H = d->H;
  p.Hkv = d->Hkv;
  p.T = d->T;
  p.Tk = d->T;
  p.delta = 0;
  p.S = d->S > 0 ? static_cast<int>(slots_in_memory(d)) : 0;  // memory stride (no depth when S = 0)
  p.S_read = d->S;
  p.d = d->d;
  p.G = d->H / d->Hkv;
  p.scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt(static_cast<float>(d->d));
  p.scale_log2 = p.scale * moda::kLog2e;
  return p;
}

bool sync_mode() {
  const char* e = std::getenv("MODA_SYNC");
  return e != nullptr && e[0] == '1';
}

int* status_word() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<int*>(ptr);
}

moda_status read_status(int clear, cudaStream_t s) {
  int* w = status_word();
  if (w == nullptr) return MODA_ERR_CUDA;
  int host = 0;
  if (cudaMemcpyAsync(&host, w, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MODA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MODA_ERR_CUDA;
  if (clear && host != 0) {
    if (cudaMemsetAsync(w, 0, sizeof(int), s) != cudaSuccess) return MODA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MODA_ERR_CUDA;
  }
  return static_cast<moda_status>(host);
}

moda_status finish(cudaError_t launch, cudaStream_t s) {
  if (launch != cudaSuccess) return MODA_ERR_CUDA;
  if (sync_mode()) {
    if (cudaStreamSynchronize(s) != cudaSuccess) return MODA_ERR_CUDA;
    return read_status(1, s);
  }
  return MODA_OK;
}

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

size_t stats_bytes(const moda_desc* d) { return align256(size_t(d->B) * d->H * d->T * 2 * sizeof(float)); }
size_t dq_accum_bytes(const moda_desc* d) {
  return align256(size_t(d->B) * d->H * d->T * d->d * sizeof(float));
}

// A key range of Tk positions whose key j is visible to query position t iff
// j <= t + delta: 0 <= delta, 1 <= Tk <= T + delta (every query sees key 0 and the last
// query sees every key).  Sets the effective (Tk, delta) of `p`: delta is clamped to Tk,
// which leaves every mask unchanged and keeps t + delta within 32 bits.
moda_status check_chunk(const moda_desc* d, int32_t Tk, int32_t delta, moda::Problem& p) {
  if (Tk < 1 || delta < 0) return MODA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(Tk) > static_cast<int64_t>(d->T) + delta) return MODA_ERR_INVALID_ARG;
  if (mul_capped(mul_capped(mul_capped(d->B, d->Hkv), Tk), d->d) > kMaxElems) return MODA_ERR_INVALID_ARG;
  const int32_t eff = delta < Tk ? delta : Tk;
  if (static_cast<int64_t>(d->T) + eff >= (int64_t(1) << 31)) return MODA_ERR_UNSUPPORTED;
  p.Tk = Tk;
  p.delta = eff;
  return MODA_OK;
}

moda_status fwd_impl(const moda_desc* desc, int32_t Tk, int32_t delta, const void* q, const void* k,
                     const void* v, const void* kd, const void* vd, void* o, float* lse, void* stream) {
  moda_status st = check_desc(desc);
  if (st != MODA_OK) return st;
  moda::FwdArgs a;
  a.p = problem_of(desc);
  st = check_chunk(desc, Tk, delta, a.p);
  if (st != MODA_OK) return st;
  if (!q || !k || !v || !o) return MODA_ERR_INVALID_ARG;
  if (desc->S > 0 && (!kd || !vd)) return MODA_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, kd, vd, static_cast<const void*>(o), static_cast<const void*>(lse)})
    if (p && !aligned16(p)) return MODA_ERR_INVALID_ARG;
  a.status = status_word();
  if (a.status == nullptr) return MODA_ERR_CUDA;
  a.q = q;
  a.k = k;
  a.v = v;
  a.kd = desc->S > 0 ? kd : nullptr;
  a.vd = desc->S > 0 ? vd : nullptr;
  a.o = o;
  a.lse = lse;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (desc->dtype == MODA_DTYPE_BF16 && moda::fwd_sm103_supported(a.p))
    e = moda::launch_fwd_sm103(a, s);
  else
    e = moda::launch_fwd_simt(a, desc->dtype, s);
  return finish(e, s);
}

}  // namespace

extern "C" {

moda_status moda_fwd(const moda_desc* desc, const void* q, const void* k, const void* v, const void* kd,
                     const void* vd, void* o, float* lse, void* stream) {
  if (desc == nullptr) return MODA_ERR_INVALID_ARG;
  return fwd_impl(desc, desc->T, 0, q, k, v, kd, vd, o, lse, stream);
}

moda_status moda_fwd_partial(const moda_desc* desc, int32_t Tk, int32_t delta, const void* q, const void* k,
                             const void* v, const void* kd, const void* vd, void* o, float* lse, void* stream) {
  if (lse == nullptr) return MODA_ERR_INVALID_ARG;  // the merge needs every partial's lse
  return fwd_impl(desc, Tk, delta, q, k, v, kd, vd, o, lse, stream);
}

size_t moda_bwd_workspace_bytes(const moda_desc* desc) {
  if (check_desc(desc) != MODA_OK) return 0;
  return stats_bytes(desc) + dq_accum_bytes(desc);
}

moda_status moda_bwd(const moda_desc* desc, const void* q, const void* k, const void* v, const void* kd,
                     const void* vd, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                     void* dv, void* dkd, void* dvd, void* workspace, size_t workspace_bytes, void* stream) {
  return moda_bwd_profiled(desc, q, k, v, kd, vd, o, lse, dout, dq, dk, dv, dkd, dvd, workspace, workspace_bytes,
                           stream, nullptr, 0);
}

}  // extern "C"

namespace {

// Backward of a chunk pair (Tk, delta as for check_chunk).  acc: dq/dk/dv are float32
// accumulators added to (dq_acc [B,H,T,d], dk_acc/dv_acc [B,Hkv,Tk,d]) instead of
// storage-type outputs.
moda_status bwd_impl(const moda_desc* desc, int32_t Tk, int32_t delta, bool acc, const void* q, const void* k,
                     const void* v, const void* kd, const void* vd, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, void* dkd, void* dvd, void* workspace,
                     size_t workspace_bytes, void* stream, void** events, int32_t n_events) {
  moda_status st = check_desc(desc);
  if (st != MODA_OK) return st;
  moda::BwdArgs a;
  a.p = problem_of(desc);
  st = check_chunk(desc, Tk, delta, a.p);
  if (st != MODA_OK) return st;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return MODA_ERR_INVALID_ARG;
  if (desc->S > 0 && (!kd || !vd || !dkd || !dvd)) return MODA_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, kd, vd, o, static_cast<const void*>(lse), dout, static_cast<const void*>(dq),
                        static_cast<const void*>(dk), static_cast<const void*>(dv), static_cast<const void*>(dkd),
                        static_cast<const void*>(dvd)})
    if (p && !aligned16(p)) return MODA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < moda_bwd_workspace_bytes(desc)) return MODA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MODA_ERR_INVALID_ARG;
  a.status = status_word();
  if (a.status == nullptr) return MODA_ERR_CUDA;
  a.q = q;
  a.k = k;
  a.v = v;
  a.kd = desc->S > 0 ? kd : nullptr;
  a.vd = desc->S > 0 ? vd : nullptr;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.dq = acc ? nullptr : dq;
  a.dk = acc ? nullptr : dk;
  a.dv = acc ? nullptr : dv;
  a.dq_acc = acc ? static_cast<float*>(dq) : nullptr;
  a.dk_acc = acc ? static_cast<float*>(dk) : nullptr;
  a.dv_acc = acc ? static_cast<float*>(dv) : nullptr;
  a.dkd = desc->S > 0 ? dkd : nullptr;
  a.dvd = desc->S > 0 ? dvd : nullptr;
  a.events = events;
  a.n_events = events != nullptr ? n_events : 0;
  a.stats = static_cast<float2*>(workspace);
  a.dq_accum = reinterpret_cast<float*>(static_cast<char*>(workspace) + stats_bytes(desc));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (desc->dtype == MODA_DTYPE_BF16 && moda::bwd_sm103_supported(a.p))
    e = moda::launch_bwd_sm103(a, s);
  else
    e = moda::launch_bwd_simt(a, desc->dtype, s);
  return finish(e, s);
}

}  // namespace

extern "C" {

moda_status moda_bwd_profiled(const moda_desc* desc, const void* q, const void* k, const void* v, const void* kd,
                              const void* vd, const void* o, const float* lse, const void* dout, void* dq, void* dk,
                              void* dv, void* dkd, void* dvd, void* workspace, size_t workspace_bytes, void* stream,
                              void** events, int32_t n_events) {
  if (desc == nullptr) return MODA_ERR_INVALID_ARG;
  return bwd_impl(desc, desc->T, 0, false, q, k, v, kd, vd, o, lse, dout, dq, dk, dv, dkd, dvd, workspace,
                  workspace_bytes, stream, events, n_events);
}

moda_status moda_bwd_partial(const moda_desc* desc, int32_t Tk, int32_t delta, const void* q, const void* k,
                             const void* v, const void* kd, const void* vd, const void* o, const float* lse,
                             const void* dout, float* dq_acc, float* dk_acc, float* dv_acc, void* dkd, void* dvd,
                             void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(desc, Tk, delta, true, q, k, v, kd, vd, o, lse, dout, dq_acc, dk_acc, dv_acc, dkd, dvd,
                  workspace, workspace_bytes, stream, nullptr, 0);
}

moda_status moda_merge_partial(const moda_desc* desc, float* o_acc, float* lse_acc, const void* o_part,
                               const float* lse_part, int32_t first, void* o_out, void* stream) {
  moda_status st = check_desc(desc);
  if (st != MODA_OK) return st;
  if (!o_acc || !lse_acc || !o_part || !lse_part) return MODA_ERR_INVALID_ARG;
  for (const void* p : {static_cast<const void*>(o_acc), static_cast<const void*>(lse_acc), o_part,
                        static_cast<const void*>(lse_part), static_cast<const void*>(o_out)})
    if (p && !aligned16(p)) return MODA_ERR_INVALID_ARG;
  moda::MergeArgs a;
  a.rows = static_cast<int64_t>(desc->B) * desc->H * desc->T;
  a.d = desc->d;
  a.first = first != 0;
  a.o_acc = o_acc;
  a.lse_acc = lse_acc;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.o_out = o_out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(moda::launch_merge(a, desc->dtype, s), s);
}

moda_status moda_convert_f32(int64_t n, const float* src, int32_t dtype, void* dst, void* stream) {
  if (n < 0 || n > kMaxElems) return MODA_ERR_INVALID_ARG;
  if (dtype != MODA_DTYPE_F32 && dtype != MODA_DTYPE_BF16) return MODA_ERR_UNSUPPORTED;
  if (n == 0) return MODA_OK;
  if (!src || !dst || !aligned16(src) || !aligned16(dst)) return MODA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(moda::launch_convert(n, src, dst, dtype, s), s);
}

size_t moda_decode_workspace_bytes(const moda_desc* desc) {
  if (check_desc(desc) != MODA_OK) return 0;
  const moda::DecodeSplit sp = moda::decode_split(problem_of(desc));
  return align256(static_cast<size_t>(sp.n_split) * desc->B * desc->H * (desc->d + 2) * sizeof(float));
}

moda_status moda_decode(const moda_desc* desc, int64_t kv_capacity, const void* q, const void* k_cache,
                        const void* v_cache, const void* kd, const void* vd, void* o, float* lse, void* workspace,
                        size_t workspace_bytes, void* stream) {
  moda_status st = check_desc(desc);
  if (st != MODA_OK) return st;
  if (desc->dtype != MODA_DTYPE_BF16) return MODA_ERR_UNSUPPORTED;
  const int64_t cap = kv_capacity > 0 ? kv_capacity : desc->T;
  if (cap < desc->T) return MODA_ERR_INVALID_ARG;
  // TMA row coordinates are 32-bit
  if (static_cast<int64_t>(desc->B) * desc->Hkv * cap >= (int64_t(1) << 31) ||
      static_cast<int64_t>(desc->B) * desc->Hkv * slots_in_memory(desc) >= (int64_t(1) << 31))
    return MODA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !o) return MODA_ERR_INVALID_ARG;
  if (desc->S > 0 && (!kd || !vd)) return MODA_ERR_INVALID_ARG;
  for (const void* p : {q, k_cache, v_cache, kd, vd, static_cast<const void*>(o), static_cast<const void*>(lse)})
    if (p && !aligned16(p)) return MODA_ERR_INVALID_ARG;
  moda::DecodeArgs a;
  a.p = problem_of(desc);
  if (!moda::decode_sm103_supported(a.p)) return MODA_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < moda_decode_workspace_bytes(desc)) return MODA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MODA_ERR_INVALID_ARG;
  a.status = status_word();
  if (a.status == nullptr) return MODA_ERR_CUDA;
  a.cap = cap;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.kd = desc->S > 0 ? kd : nullptr;
  a.vd = desc->S > 0 ? vd : nullptr;
  a.o = o;
  a.lse = lse;
  a.part = static_cast<float*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(moda::launch_decode_sm103(a, s), s);
}

moda_status moda_depth_store_kv(const moda_desc* desc, int32_t slot, const void* k, const void* v, void* kd,
                                void* vd, void* stream) {
  moda_status st = check_desc(desc);
  if (st != MODA_OK) return st;
  if (desc->dtype != MODA_DTYPE_BF16) return MODA_ERR_UNSUPPORTED;
  const int64_t n_slots = slots_in_memory(desc);
  if (n_slots < 1 || slot < 0 || slot >= n_slots) return MODA_ERR_INVALID_ARG;
  if (!k || !v || !kd || !vd) return MODA_ERR_INVALID_ARG;
  for (const void* p : {k, v, static_cast<const void*>(kd), static_cast<const void*>(vd)})
    if (!aligned16(p)) return MODA_ERR_INVALID_ARG;
  moda::DepthWriteArgs a{};
  a.B = desc->B;
  a.Hkv = desc->Hkv;
  a.T = desc->T;
  a.S = static_cast<int>(n_slots);
  a.d = desc->d;
  a.slot = slot;
  a.k = k;
  a.v = v;
  a.kd = kd;
  a.vd = vd;
  a.status = status_word();
  if (a.status == nullptr) return MODA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(moda::launch_depth_store_sm103(a, s), s);
}

moda_status moda_depth_project_kv(const moda_desc* desc, int32_t slot, int32_t d_model, const void* x,
                                  const void* wk, const void* wv, void* kd, void* vd, void* stream) {
  moda_status st = check_desc(desc);
  if (st != MODA_OK) return st;
  if (desc->dtype != MODA_DTYPE_BF16) return MODA_ERR_UNSUPPORTED;
  const int64_t n_slots = slots_in_memory(desc);
  if (n_slots < 1 || slot < 0 || slot >= n_slots) return MODA_ERR_INVALID_ARG;
  if (d_model < 8 || d_model % 8 != 0) return MODA_ERR_INVALID_ARG;  // 16-byte row strides
  if ((desc->Hkv * desc->d) % 64 != 0) return MODA_ERR_UNSUPPORTED;
  if (desc->B > 65535 || (desc->T + 127) / 128 > 65535) return MODA_ERR_UNSUPPORTED;  // grid limits
  if (mul_capped(mul_capped(desc->B, desc->T), d_model) > kMaxElems) return MODA_ERR_INVALID_ARG;
  if (!x || !wk || !wv || !kd || !vd) return MODA_ERR_INVALID_ARG;
  for (const void* p : {x, wk, wv, static_cast<const void*>(kd), static_cast<const void*>(vd)})
    if (!aligned16(p)) return MODA_ERR_INVALID_ARG;
  moda::DepthWriteArgs a{};
  a.B = desc->B;
  a.Hkv = desc->Hkv;
  a.T = desc->T;
  a.S = static_cast<int>(n_slots);
  a.d = desc->d;
  a.slot = slot;
  a.Dm = d_model;
  a.x = x;
  a.wk = wk;
  a.wv = wv;
  a.kd = kd;
  a.vd = vd;
  a.status = status_word();
  if (a.status == nullptr) return MODA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(moda::launch_depth_project_sm103(a, s), s);
}

moda_status moda_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* w = status_word();
  if (w == nullptr) return MODA_ERR_CUDA;
  // leave no earlier error behind that would mask the result
  moda_status before = read_status(1, s);
  if (before == MODA_ERR_CUDA) return MODA_ERR_CUDA;
  const uint64_t lim = limit_ns < 1000000ull ? 1000000ull : (limit_ns > 2000000000ull ? 2000000000ull : limit_ns);
  if (moda::launch_wait_selftest(w, lim, s) != cudaSuccess) return MODA_ERR_CUDA;
  return read_status(1, s);
}

moda_status moda_device_status(int clear, void* stream) {
  return read_status(clear, static_cast<cudaStream_t>(stream));
}

const char* moda_status_str(moda_status status) {
  switch (status) {
    case MODA_OK: return "MODA_OK";
    case MODA_ERR_INVALID_ARG: return "MODA_ERR_INVALID_ARG";
    case MODA_ERR_UNSUPPORTED: return "MODA_ERR_UNSUPPORTED";
    case MODA_ERR_CUDA: return "MODA_ERR_CUDA";
    case MODA_ERR_TIMEOUT: return "MODA_ERR_TIMEOUT";
    case MODA_ERR_WORKSPACE: return "MODA_ERR_WORKSPACE";
  }
  return "MODA_ERR_UNKNOWN";
}

int32_t moda_version(void) { return 100; }

int64_t moda_launch_count(void) { return moda::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
