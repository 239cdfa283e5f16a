// MoDA on the CUDA cores: the float32 forward and backward (and the portable
// kernels the backward preprocess shares with the tensor-core path).
//
// One warp owns one query row (or one key / one position in the backward); lane
// l holds columns [l*N, l*N+N) of every d-vector (N = d/32), so each row load is
// one coalesced 8/16-byte access per lane and a score is a 5-step xor-shuffle
// reduction.  Scores carry the log2(e)-folded scale so every exponential is
// exp2 (slides' Algorithm 1 writes 2^(S-m); backup frame "pseudocode needs
// implementation-level checks" gives the log2(e) correction).
//
// Forward state per row follows the frame "Shared online-softmax states preserve
// the joint operator": running max m, denominator acc, numerator o, updated key
// by key over the causal sequence keys and then the S depth slots of the same
// position, normalised once at the end.  Key j is visible to position t when
// j <= t + delta and j < Tk (delta = 0, Tk = T for a whole sequence; a key chunk of
// an earlier range of positions has delta > 0).
#include "moda_common.cuh"

namespace moda {
namespace {

constexpr int kWarps = 8;  // rows (keys, positions) per CTA

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int N>
__device__ __forceinline__ void load_frag(const float* p, float (&x)[N]) {
  if constexpr (N == 4) {
    float4 u = __ldg(reinterpret_cast<const float4*>(p));
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
  } else {
    static_assert(N == 2, "d must be 64 or 128");
    float2 u = __ldg(reinterpret_cast<const float2*>(p));
    x[0] = u.x; x[1] = u.y;
  }
}

template <int N>
__device__ __forceinline__ void load_frag(const __nv_bfloat16* p, float (&x)[N]) {
  if constexpr (N == 4) {
    uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.x));
    float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    static_assert(N == 2, "d must be 64 or 128");
    unsigned int u = __ldg(reinterpret_cast<const unsigned int*>(p));
    float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
    x[0] = a.x; x[1] = a.y;
  }
}

template <typename T, int N>
__device__ __forceinline__ void store_frag(T* p, const float (&x)[N]) {
#pragma unroll
  for (int c = 0; c < N; ++c) p[c] = from_f32<T>(x[c]);
}

// Adds a fragment to a float32 accumulator (the accumulating backward of a chunk pair).
template <int N>
__device__ __forceinline__ void add_frag(float* p, const float (&x)[N]) {
#pragma unroll
  for (int c = 0; c < N; ++c) p[c] += x[c];
}

template <int N>
__device__ __forceinline__ float dot(const float (&a)[N], const float (&b)[N]) {
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < N; ++c) s = fmaf(a[c], b[c], s);
  return s;
}

// Online update of (m, acc, o) with one key of log2-domain score s2 and value vf.
template <int N>
__device__ __forceinline__ void online_update(float s2, const float (&vf)[N], float& m, float& acc,
                                              float (&o)[N]) {
  const float mn = fmaxf(m, s2);
  const float corr = exp2f(m - mn);  // m = -inf on the first key: corr = 0
  const float pj = exp2f(s2 - mn);
  acc = fmaf(acc, corr, pj);
#pragma unroll
  for (int c = 0; c < N; ++c) o[c] = fmaf(o[c], corr, pj * vf[c]);
  m = mn;
}

// ---------------------------------------------------------------- forward
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) fwd_simt_kernel(const FwdArgs a) {
  constexpr int N = D / 32;
  const Problem& p = a.p;
  const int lane = threadIdx.x & 31;
  const int tiles = (p.T + kWarps - 1) / kWarps;
  const int64_t bh = blockIdx.x / tiles;
  const int t = (blockIdx.x % tiles) * kWarps + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H), g = h / p.G;
  const int64_t bg = static_cast<int64_t>(b) * p.Hkv + g;
  const T* q = static_cast<const T*>(a.q) + (bh * p.T + t) * D + lane * N;
  const T* k = static_cast<const T*>(a.k) + bg * p.Tk * D + lane * N;
  const T* v = static_cast<const T*>(a.v) + bg * p.Tk * D + lane * N;
  const int j_end = min(t + p.delta, p.Tk - 1);  // last visible key

  float qf[N], kf[N], vf[N], o[N];
  load_frag(q, qf);
#pragma unroll
  for (int c = 0; c < N; ++c) {
    qf[c] *= p.scale_log2;
    o[c] = 0.f;
  }
  float m = -INFINITY, acc = 0.f;
  // causal sequence keys j <= t + delta (j < Tk)
  for (int j = 0; j <= j_end; ++j) {
    load_frag(k + static_cast<int64_t>(j) * D, kf);
    const float s2 = warp_sum(dot(qf, kf));
    load_frag(v + static_cast<int64_t>(j) * D, vf);
    online_update(s2, vf, m, acc, o);
  }
  // same-position depth slots, same (m, acc, o) state
  if (p.S > 0) {
    const int64_t slab = (bg * p.T + t) * p.S * D + lane * N;
    const T* kd = static_cast<const T*>(a.kd) + slab;
    const T* vd = static_cast<const T*>(a.vd) + slab;
    for (int i = 0; i < p.S_read; ++i) {
      load_frag(kd + static_cast<int64_t>(i) * D, kf);
      const float s2 = warp_sum(dot(qf, kf));
      load_frag(vd + static_cast<int64_t>(i) * D, vf);
      online_update(s2, vf, m, acc, o);
    }
  }
  const float inv = 1.f / acc;
#pragma unroll
  for (int c = 0; c < N; ++c) o[c] *= inv;
  store_frag(static_cast<T*>(a.o) + (bh * p.T + t) * D + lane * N, o);
  if (a.lse != nullptr && lane == 0) a.lse[bh * p.T + t] = (m + log2f(acc)) * kLn2;
}

// ---------------------------------------------------------------- backward
// Row statistics for every row (b, h, t): {-lse * log2(e), Delta_t = dout_t . o_t}.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_delta_kernel(const BwdArgs a) {
  constexpr int N = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t rows = static_cast<int64_t>(a.p.B) * a.p.H * a.p.T;
  if (row >= rows) return;
  float of[N], df[N];
  load_frag(static_cast<const T*>(a.o) + row * D + lane * N, of);
  load_frag(static_cast<const T*>(a.dout) + row * D + lane * N, df);
  const float s = warp_sum(dot(of, df));
  if (lane == 0) a.stats[row] = make_float2(-a.lse[row] * kLog2e, s);
}

// dq for one row: sequence keys j <= t, then the depth slots of position t.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_simt_kernel(const BwdArgs a) {
  constexpr int N = D / 32;
  const Problem& p = a.p;
  const int lane = threadIdx.x & 31;
  const int tiles = (p.T + kWarps - 1) / kWarps;
  const int64_t bh = blockIdx.x / tiles;
  const int t = (blockIdx.x % tiles) * kWarps + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H), g = h / p.G;
  const int64_t bg = static_cast<int64_t>(b) * p.Hkv + g;
  const int64_t row = bh * p.T + t;
  const T* k = static_cast<const T*>(a.k) + bg * p.Tk * D + lane * N;
  const T* v = static_cast<const T*>(a.v) + bg * p.Tk * D + lane * N;
  const int j_end = min(t + p.delta, p.Tk - 1);
  float qf[N], df[N], kf[N], vf[N], dq[N];
  load_frag(static_cast<const T*>(a.q) + row * D + lane * N, qf);
  load_frag(static_cast<const T*>(a.dout) + row * D + lane * N, df);
#pragma unroll
  for (int c = 0; c < N; ++c) {
    qf[c] *= p.scale_log2;
    dq[c] = 0.f;
  }
  const float2 st = a.stats[row];
  const float lse2 = -st.x;
  const float Dt = st.y;
  for (int j = 0; j <= j_end; ++j) {
    load_frag(k + static_cast<int64_t>(j) * D, kf);
    load_frag(v + static_cast<int64_t>(j) * D, vf);
    const float pj = exp2f(warp_sum(dot(qf, kf)) - lse2);
    const float ds = pj * (warp_sum(dot(df, vf)) - Dt);
#pragma unroll
    for (int c = 0; c < N; ++c) dq[c] = fmaf(ds, kf[c], dq[c]);
  }
  if (p.S > 0) {
    const int64_t slab = (bg * p.T + t) * p.S * D + lane * N;
    const T* kd = static_cast<const T*>(a.kd) + slab;
    const T* vd = static_cast<const T*>(a.vd) + slab;
    for (int i = 0; i < p.S_read; ++i) {
      load_frag(kd + static_cast<int64_t>(i) * D, kf);
      load_frag(vd + static_cast<int64_t>(i) * D, vf);
      const float pj = exp2f(warp_sum(dot(qf, kf)) - lse2);
      const float ds = pj * (warp_sum(dot(df, vf)) - Dt);
#pragma unroll
      for (int c = 0; c < N; ++c) dq[c] = fmaf(ds, kf[c], dq[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < N; ++c) dq[c] *= p.scale;
  if (a.dq_acc != nullptr) add_frag(a.dq_acc + row * D + lane * N, dq);
  else store_frag(static_cast<T*>(a.dq) + row * D + lane * N, dq);
}

// dk, dv for one sequence key (b, g, j): every row t >= j - delta of the G heads of g.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dkdv_simt_kernel(const BwdArgs a) {
  constexpr int N = D / 32;
  const Problem& p = a.p;
  const int lane = threadIdx.x & 31;
  const int tiles = (p.Tk + kWarps - 1) / kWarps;
  const int64_t bg = blockIdx.x / tiles;
  const int j = (blockIdx.x % tiles) * kWarps + (threadIdx.x >> 5);
  if (j >= p.Tk) return;
  const int b = static_cast<int>(bg / p.Hkv), g = static_cast<int>(bg % p.Hkv);
  const int t0 = max(j - p.delta, 0);  // first query position that sees key j
  float kf[N], vf[N], qf[N], df[N], dk[N], dv[N];
  load_frag(static_cast<const T*>(a.k) + (bg * p.Tk + j) * D + lane * N, kf);
  load_frag(static_cast<const T*>(a.v) + (bg * p.Tk + j) * D + lane * N, vf);
#pragma unroll
  for (int c = 0; c < N; ++c) dk[c] = dv[c] = 0.f;
  for (int hh = 0; hh < p.G; ++hh) {
    const int64_t bh = static_cast<int64_t>(b) * p.H + g * p.G + hh;
    for (int t = t0; t < p.T; ++t) {
      const int64_t row = bh * p.T + t;
      load_frag(static_cast<const T*>(a.q) + row * D + lane * N, qf);
      load_frag(static_cast<const T*>(a.dout) + row * D + lane * N, df);
      const float2 st = a.stats[row];
      const float pj = exp2f(warp_sum(dot(qf, kf)) * p.scale_log2 + st.x);
      const float ds = pj * (warp_sum(dot(df, vf)) - st.y);
#pragma unroll
      for (int c = 0; c < N; ++c) {
        dk[c] = fmaf(ds, qf[c], dk[c]);
        dv[c] = fmaf(pj, df[c], dv[c]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < N; ++c) dk[c] *= p.scale;
  if (a.dk_acc != nullptr) {
    add_frag(a.dk_acc + (bg * p.Tk + j) * D + lane * N, dk);
    add_frag(a.dv_acc + (bg * p.Tk + j) * D + lane * N, dv);
  } else {
    store_frag(static_cast<T*>(a.dk) + (bg * p.Tk + j) * D + lane * N, dk);
    store_frag(static_cast<T*>(a.dv) + (bg * p.Tk + j) * D + lane * N, dv);
  }
}

// dkd, dvd for one position (b, g, t): the G heads of g at position t.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_depth_simt_kernel(const BwdArgs a) {
  constexpr int N = D / 32;
  const Problem& p = a.p;
  const int lane = threadIdx.x & 31;
  const int tiles = (p.T + kWarps - 1) / kWarps;
  const int64_t bg = blockIdx.x / tiles;
  const int t = (blockIdx.x % tiles) * kWarps + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int b = static_cast<int>(bg / p.Hkv), g = static_cast<int>(bg % p.Hkv);
  const int64_t slab = (bg * p.T + t) * p.S * D + lane * N;
  float kf[N], vf[N], qf[N], df[N], dk[N], dv[N];
  for (int i = 0; i < p.S_read; ++i) {
    load_frag(static_cast<const T*>(a.kd) + slab + static_cast<int64_t>(i) * D, kf);
    load_frag(static_cast<const T*>(a.vd) + slab + static_cast<int64_t>(i) * D, vf);
#pragma unroll
    for (int c = 0; c < N; ++c) dk[c] = dv[c] = 0.f;
    for (int hh = 0; hh < p.G; ++hh) {
      const int64_t row = (static_cast<int64_t>(b) * p.H + g * p.G + hh) * p.T + t;
      load_frag(static_cast<const T*>(a.q) + row * D + lane * N, qf);
      load_frag(static_cast<const T*>(a.dout) + row * D + lane * N, df);
      const float2 st = a.stats[row];
      const float pj = exp2f(warp_sum(dot(qf, kf)) * p.scale_log2 + st.x);
      const float ds = pj * (warp_sum(dot(df, vf)) - st.y);
#pragma unroll
      for (int c = 0; c < N; ++c) {
        dk[c] = fmaf(ds, qf[c], dk[c]);
        dv[c] = fmaf(pj, df[c], dv[c]);
      }
    }
#pragma unroll
    for (int c = 0; c < N; ++c) dk[c] *= p.scale;
    store_frag(static_cast<T*>(a.dkd) + slab + static_cast<int64_t>(i) * D, dk);
    store_frag(static_cast<T*>(a.dvd) + slab + static_cast<int64_t>(i) * D, dv);
  }
  // slots in memory that are not read have zero gradient
#pragma unroll
  for (int c = 0; c < N; ++c) dk[c] = 0.f;
  for (int i = p.S_read; i < p.S; ++i) {
    store_frag(static_cast<T*>(a.dkd) + slab + static_cast<int64_t>(i) * D, dk);
    store_frag(static_cast<T*>(a.dvd) + slab + static_cast<int64_t>(i) * D, dk);
  }
}

unsigned blocks_for(int64_t groups, int T) { return static_cast<unsigned>(groups * ((T + kWarps - 1) / kWarps)); }

template <typename T, int D>
cudaError_t fwd_simt(const FwdArgs& a, cudaStream_t s) {
  const unsigned grid = blocks_for(static_cast<int64_t>(a.p.B) * a.p.H, a.p.T);
  fwd_simt_kernel<T, D><<<grid, kWarps * 32, 0, s>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_simt(const BwdArgs& a, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.p.B) * a.p.H * a.p.T;
  mark_event(a, 0, s);
  bwd_delta_kernel<T, D><<<static_cast<unsigned>((rows + kWarps - 1) / kWarps), kWarps * 32, 0, s>>>(a);
  mark_event(a, 1, s);
  mark_event(a, 2, s);
  if (a.p.S > 0)
    bwd_depth_simt_kernel<T, D>
        <<<blocks_for(static_cast<int64_t>(a.p.B) * a.p.Hkv, a.p.T), kWarps * 32, 0, s>>>(a);
  mark_event(a, 3, s);
  mark_event(a, 4, s);
  bwd_dkdv_simt_kernel<T, D><<<blocks_for(static_cast<int64_t>(a.p.B) * a.p.Hkv, a.p.Tk), kWarps * 32, 0, s>>>(a);
  mark_event(a, 5, s);
  mark_event(a, 6, s);
  bwd_dq_simt_kernel<T, D><<<blocks_for(static_cast<int64_t>(a.p.B) * a.p.H, a.p.T), kWarps * 32, 0, s>>>(a);
  mark_event(a, 7, s);
  count_launches(a.p.S > 0 ? 4 : 3);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& a, int dtype, cudaStream_t s) {
  if (dtype == 0) return a.p.d == 64 ? fwd_simt<float, 64>(a, s) : fwd_simt<float, 128>(a, s);
  return a.p.d == 64 ? fwd_simt<__nv_bfloat16, 64>(a, s) : fwd_simt<__nv_bfloat16, 128>(a, s);
}

cudaError_t launch_bwd_delta(const BwdArgs& a, int dtype, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.p.B) * a.p.H * a.p.T;
  const unsigned grid = static_cast<unsigned>((rows + kWarps - 1) / kWarps);
  if (dtype == 0) {
    if (a.p.d == 64) bwd_delta_kernel<float, 64><<<grid, kWarps * 32, 0, s>>>(a);
    else bwd_delta_kernel<float, 128><<<grid, kWarps * 32, 0, s>>>(a);
  } else {
    if (a.p.d == 64) bwd_delta_kernel<__nv_bfloat16, 64><<<grid, kWarps * 32, 0, s>>>(a);
    else bwd_delta_kernel<__nv_bfloat16, 128><<<grid, kWarps * 32, 0, s>>>(a);
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const BwdArgs& a, int dtype, cudaStream_t s) {
  if (dtype == 0) return a.p.d == 64 ? bwd_simt<float, 64>(a, s) : bwd_simt<float, 128>(a, s);
  return a.p.d == 64 ? bwd_simt<__nv_bfloat16, 64>(a, s) : bwd_simt<__nv_bfloat16, 128>(a, s);
}

}  // namespace moda
