// MoDA decode step for bf16 on sm_103a.  For every (batch, query head) the query of the
// newest position T-1 attends to the sequence cache (keys 0 .. T-1, itself included) and
// to the S depth slots of its own position, under one softmax ("Mixture-of-Depths
// Attention", frame "One denominator allocates probability across both memories"; the
// decode cache of the Table 1 frame "Depth compute still accumulates quadratically in
// depth").
//
// The step is bound by HBM: each cached K/V row is read once for the G query heads of
// its kv head.  The keys are split (flash-decoding): CTA (split, b*Hkv + g) streams its
// key range in sub-tiles of 128 keys through one K and one V slot (TMA, 128-byte swizzle,
// K of the next sub-tile loading while P V of this one runs); the extra
// last split of each (b, g) takes the S depth slots.  Per sub-tile, the scores of the G
// heads are one tensor-core product S^T = K q^T (M = 128 keys, N = 16 with the heads past
// G zero, into 16 TMEM columns), read back with lane = key; the sub-tile's maximum of
// each head over all its keys sets the running max; P V is a second product, O^T = V^T
// P^T (M = 128 channels, N = 16, P^T as bf16 in shared memory), read back with lane =
// channel and added into the thread's numerators with the heads' rescale factors.  The
// CTA writes one partial state {max, sum, numerator} per head to a float32 workspace.  A second kernel
// merges the splits of each (b, h) by the same online rule and divides once.
//
// All waits are bounded (sm103_ptx.cuh); a timeout records MODA_ERR_TIMEOUT.
#include <cudaTypedefs.h>

#include <algorithm>

#include "moda_common.cuh"
#include "sm103_ptx.cuh"

namespace moda {
namespace {

using namespace sm103;

constexpr int kDecKeys = 128;    // keys per sub-tile: 4 warps x 32 lanes (per head group)
constexpr int kDecMaxG = 8;

// Threads of a CTA: 128, thread t = TMEM lane t (key t of a sub-tile for the scores,
// channel t for P V).
constexpr int kDecThreads = 128;

template <int D>
struct DecCfg {
  static constexpr int TILE_BYTES = kDecKeys * D * 2;  // one K (or V) sub-tile, bf16
  // One V slot and one K slot, each with a barrier of its own, and many resident CTAs
  // (three per SM at d = 128, six at d = 64): the other CTAs on the SM hide each one's
  // loads, and K of the next sub-tile loads while this one's softmax and P V run.  V
  // comes first: at d = 64 the P V product reads 128 rows of V^T, the last 64 of which
  // (from the K slot behind it) give output lanes that are never used.
  static constexpr int OFF_V = 0, OFF_K = TILE_BYTES;
  // q of the heads as the B operand of the score product: bf16 [16 rows][D] (rows past G
  // zero), D/64 blocks of [16 rows x 128 B], 128-byte swizzle
  static constexpr int OFF_Q = 2 * TILE_BYTES;
  static constexpr int Q_BYTES = 16 * D * 2;
  // P^T of a sub-tile as the B operand of P V: bf16 [16 rows (heads)][128 keys], keys
  // [0, 64) then [64, 128) as two blocks of [16 rows x 128 B], 128-byte swizzle
  static constexpr int OFF_PT = OFF_Q + Q_BYTES;
  static constexpr int PT_BYTES = 16 * kDecKeys * 2;
  // per-warp maxima of a sub-tile, float [4 warps][kDecMaxG]; per-warp denominators at
  // the end
  static constexpr int OFF_WM = OFF_PT + PT_BYTES;
  static constexpr int OFF_BAR = OFF_WM + 4 * kDecMaxG * 4;  // k_full, v_full, s_done, pv_done, drain
  static constexpr int SMEM = OFF_BAR + 5 * 8 + 16;
  // TMEM: S^T [0, 16) (lane = key, column = head), the sub-tile's P V [16, 32) (lane =
  // channel, column = head)
  static constexpr uint32_t TM_COLS = 32, TM_S = 0, TM_PV = 16;
};

struct DecParams {
  int B, H, Hkv, T, S, G;
  int S_read;  // depth slots read (of the S in memory per (b, g))
  int n_seq;   // sequence splits (the depth split, when S > 0, is index n_seq)
  int chunk;   // sequence keys per split, a multiple of kDecKeys
  int64_t cap; // positions allocated per (b, g) in the sequence cache
  float scale_log2;
  const __nv_bfloat16* q;
  float* part;  // [n_split][B*H][D + 2]: {max (log2 units), sum, numerator[D]}
  int* status;
};

template <int D, int HG>
__global__ void __launch_bounds__(kDecThreads, 1)
    moda_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmKd, const __grid_constant__ CUtensorMap tmVd,
                       const DecParams p) {
  using C = DecCfg<D>;
  constexpr int CH = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = threadIdx.x;  // key of a sub-tile (scores), channel (P V)
  const int split = blockIdx.x, bg = blockIdx.y;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const bool depth = split == p.n_seq;
  const int k0 = depth ? 0 : split * p.chunk;
  const int k1 = depth ? p.S_read : min(p.T, k0 + p.chunk);
  const int n_keys = max(0, k1 - k0);
  const int n_sub = (n_keys + kDecKeys - 1) / kDecKeys;
  const CUtensorMap* mk = depth ? &tmKd : &tmK;
  const CUtensorMap* mv = depth ? &tmVd : &tmV;
  const int row0 = depth ? bg * p.S : static_cast<int>(bg * p.cap) + k0;  // host checks the int range

  // K of sub-tile s + 1 is loaded once the score product of sub-tile s has read K, while
  // the softmax and P V of s still run; V of s + 1 once the P V product of s has read V
  uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* v_full = k_full + 1;
  uint64_t* s_done = k_full + 2;   // the score product of the current sub-tile is complete
  uint64_t* pv_done = k_full + 3;  // its P V product is complete
  uint64_t* drain = k_full + 4;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 5 * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 5 * 8 + 4);
  float* wm = reinterpret_cast<float*>(smem + C::OFF_WM);  // [4][kDecMaxG]

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    mbar_init(v_full, 1);
    mbar_init(s_done, 1);
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // q of the heads, bf16, rows past G zero: 16-byte chunk x of row hh
  for (int i = threadIdx.x; i < 16 * CH; i += kDecThreads) {
    const int hh = i / CH, x = i % CH;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (hh < p.G) v = *reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(b) * p.H + g * p.G + hh) * D + x * 8);
    st_shared_v4(sbase + C::OFF_Q + (x >> 3) * (16 * 128) + hh * 128 + (((x & 7) ^ (hh & 7)) << 4), v);
  }
  // P^T rows of heads past G stay zero
  for (int i = threadIdx.x; i < C::PT_BYTES / 16; i += kDecThreads)
    st_shared_v4(sbase + C::OFF_PT + i * 16, make_uint4(0, 0, 0, 0));
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_tm = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's lanes
  // the score product: A = the K sub-tile (keys x D, K-major), B = q (16 rows x D, K-major)
  constexpr uint32_t IDESC_S = idesc_bf16(kDecKeys, 16, false);
  const uint64_t k_desc = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
  const uint64_t q_desc = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
  // the P V product (O^T = V^T P^T): A = V^T (128 channels x keys, channels contiguous,
  // 64-channel blocks 16 KB apart), B = P^T (16 rows x keys, K-major)
  constexpr uint32_t IDESC_PV = idesc_bf16(128, 16, false) | (1u << 15);  // A M-major
  const uint64_t v_desc = sdesc_sw128(sbase + C::OFF_V, kDecKeys * 128, 1024);
  const uint64_t pt_desc = sdesc_sw128(sbase + C::OFF_PT, 16, 1024);

  // K (kind 0) or V (kind 1) of sub-tile s into its slot
  auto issue = [&](int s, int kind) {
    uint8_t* dst = smem + (kind ? C::OFF_V : C::OFF_K);
    uint64_t* bar = kind ? v_full : k_full;
    mbar_arrive_expect_tx(bar, C::TILE_BYTES);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_load_2d(dst + h * (kDecKeys * 128), kind ? mv : mk, bar, h * 64, row0 + s * kDecKeys);
  };
  if (threadIdx.x == 0) {
    prefetch_tmap(mk);
    prefetch_tmap(mv);
    if (n_sub > 0) {
      issue(0, 0);
      issue(0, 1);
    }
  }

  // The split's state per head: the running max (the same in every thread), this thread's
  // part of the denominator (over its keys) and, for channel r, the numerator.
  float m[HG], l[HG], o[HG];
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
    o[hh] = 0.f;
  }
  int issued_k = min(n_sub, 1), issued_v = issued_k;  // sub-tiles whose K / V loads are issued
  int mma_issued = 0;                                  // products issued (thread 0)
  bool failed = false;
  for (int s = 0; s < n_sub; ++s) {
    const uint32_t par = s & 1;
    if (__syncthreads_or(!mbar_wait(k_full, par, abort_flag))) {  // block-uniform
      failed = true;
      break;
    }
    const int base_key = s * kDecKeys;
    // ---- scores of the heads for the sub-tile's keys on the tensor core
    if (threadIdx.x == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16_ss(tmem + C::TM_S, sdesc_add(k_desc, (kk >> 2) * (kDecKeys * 128) + (kk & 3) * 32),
                    sdesc_add(q_desc, (kk >> 2) * (16 * 128) + (kk & 3) * 32), IDESC_S, kk > 0);
      mma_commit(s_done);
      ++mma_issued;
    }
    if (__syncthreads_or(!mbar_wait(s_done, par, abort_flag))) {
      failed = true;
      break;
    }
    tc_fence_after();
    uint32_t sv[16];
    tmem_ld16(lane_tm + C::TM_S, sv);  // lane = key r, column = head
    tc_fence_before();
    // the product has read K: load the next sub-tile's K
    if (threadIdx.x == 0 && issued_k < n_sub) issue(issued_k, 0);
    ++issued_k;
    const bool valid = base_key + r < n_keys;
    float sc[HG];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      sc[hh] = valid ? __uint_as_float(sv[hh]) * p.scale_log2 : -INFINITY;
      float w = sc[hh];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, off));
      if (lane == 0) wm[warp * kDecMaxG + hh] = w;
    }
    __syncthreads();
    // ---- online softmax with the sub-tile's maximum over all four warps
    float corr[HG];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      const float cmax = fmaxf(fmaxf(wm[hh], wm[kDecMaxG + hh]), fmaxf(wm[2 * kDecMaxG + hh], wm[3 * kDecMaxG + hh]));
      const float m_new = fmaxf(m[hh], cmax);
      corr[hh] = (m[hh] == -INFINITY) ? 0.f : ex2(m[hh] - m_new);
      const float pr = valid ? ex2(sc[hh] - m_new) : 0.f;
      l[hh] = l[hh] * corr[hh] + pr;
      m[hh] = m_new;
      // P^T[hh][r] (bf16) for the P V product
      const __nv_bfloat16 pb = __float2bfloat16_rn(pr);
      const uint32_t addr = sbase + C::OFF_PT + (r >> 6) * (16 * 128) + hh * 128 +
                            ((((r & 63) >> 3) ^ (hh & 7)) << 4) + (r & 7) * 2;
      asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(*reinterpret_cast<const unsigned short*>(&pb))
                   : "memory");
    }
    if (__syncthreads_or(!mbar_wait(v_full, par, abort_flag))) {
      failed = true;
      break;
    }
    if (!valid) {
      // rows past the keys read (a cache's positions past T, a ring's unread slots) may
      // hold anything, NaN included: they enter the product with P = 0, so make them zero
#pragma unroll
      for (int x = 0; x < CH; ++x)
        st_shared_v4(sbase + C::OFF_V + (x >> 3) * (kDecKeys * 128) + r * 128 + ((x & 7) << 4), make_uint4(0, 0, 0, 0));
    }
    fence_proxy_async_smem();
    __syncthreads();
    // ---- P V on the tensor core: O^T of the sub-tile (lane = channel, column = head)
    if (threadIdx.x == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kDecKeys / 16; ++kk)
        mma_bf16_ss(tmem + C::TM_PV, sdesc_add(v_desc, kk * 2048),
                    sdesc_add(pt_desc, (kk >> 2) * (16 * 128) + (kk & 3) * 32), IDESC_PV, kk > 0);
      mma_commit(pv_done);
      ++mma_issued;
    }
    if (__syncthreads_or(!mbar_wait(pv_done, par, abort_flag))) {
      failed = true;
      break;
    }
    tc_fence_after();
    uint32_t pv[16];
    tmem_ld16(lane_tm + C::TM_PV, pv);
    tc_fence_before();
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) o[hh] = o[hh] * corr[hh] + __uint_as_float(pv[hh]);
    // the product has read V and P^T: load the next sub-tile's V
    if (threadIdx.x == 0 && issued_v < n_sub) issue(issued_v, 1);
    ++issued_v;
  }
  if (failed && threadIdx.x == 0) {
    record_status(p.status, kStatusTimeout);
    // let the copies and products still in flight land before the CTA exits
    volatile int never = 0;
    if (issued_k > 0 && issued_k <= n_sub) mbar_wait(k_full, (issued_k - 1) & 1, &never);
    if (issued_v > 0 && issued_v <= n_sub) mbar_wait(v_full, (issued_v - 1) & 1, &never);
    if (mma_issued > 0) {
      mma_commit(drain);
      mbar_wait(drain, 0, &never);
    }
  }
  // every product has been read (the waits above): TMEM is no longer needed
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
  if (failed) return;
  // ---- this split's state: {max, denominator, numerator[D]} per head
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    float ls = l[hh];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    if (lane == 0) wm[warp * kDecMaxG + hh] = ls;
  }
  __syncthreads();
  const int64_t row_base = static_cast<int64_t>(split) * p.B * p.H + static_cast<int64_t>(b) * p.H + g * p.G;
  for (int hh = 0; hh < p.G && hh < HG; ++hh) {
    float* dst = p.part + (row_base + hh) * (D + 2);
    if (r < D) dst[2 + r] = o[hh];
    if (r == 0) {
      dst[0] = m[hh];
      dst[1] = wm[hh] + wm[kDecMaxG + hh] + wm[2 * kDecMaxG + hh] + wm[3 * kDecMaxG + hh];
    }
  }
}

struct DecMergeParams {
  int BH, n_split;
  const float* part;
  __nv_bfloat16* o;
  float* lse;  // may be null
};

// One warp per (b, h): merge the splits' partial states by the online rule, divide once.
// The splits' maxima are read one per lane (32 splits at a time) and reduced by shuffles;
// each lane then weighs its splits' denominators, and the numerators are read four
// splits at a time, so the loads of a warp do not wait on one another.
template <int D>
__global__ void __launch_bounds__(128) moda_decode_merge_kernel(const DecMergeParams p) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= p.BH) return;
  auto state = [&](int sp) { return p.part + (static_cast<int64_t>(sp) * p.BH + row) * (D + 2); };
  float mx = -INFINITY;
  for (int s0 = 0; s0 < p.n_split; s0 += 32)
    if (s0 + lane < p.n_split) mx = fmaxf(mx, state(s0 + lane)[0]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float L = 0.f;
  for (int s0 = 0; s0 < p.n_split; s0 += 32) {
    if (s0 + lane < p.n_split) {
      const float* ps = state(s0 + lane);
      const float ms = ps[0];
      if (ms != -INFINITY) L += ps[1] * ex2(ms - mx);  // a split without keys has ms = -inf
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  int sp = 0;
  for (; sp + 4 <= p.n_split; sp += 4) {
    float ms[4], v[4][CPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float* ps = state(sp + u);
      ms[u] = ps[0];
#pragma unroll
      for (int c = 0; c < CPL; ++c) v[u][c] = ps[2 + lane * CPL + c];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (ms[u] == -INFINITY) continue;
      const float w = ex2(ms[u] - mx);
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[c] += v[u][c] * w;
    }
  }
  for (; sp < p.n_split; ++sp) {
    const float* ps = state(sp);
    const float ms = ps[0];
    if (ms == -INFINITY) continue;
    const float w = ex2(ms - mx);
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] += ps[2 + lane * CPL + c] * w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* orow = p.o + row * D + lane * CPL;
#pragma unroll
  for (int c = 0; c < CPL; ++c) orow[c] = __float2bfloat16_rn(acc[c] * inv);
  if (p.lse != nullptr && lane == 0) p.lse[row] = (mx + __log2f(L)) * kLn2;
}

// ---------------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 dec_encode_fn() {
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
}

// bf16 rows [rows][D] as the 2-D tensor (D, rows), box 64 x kDecKeys, 128-byte swizzle.
bool dec_map(CUtensorMap* map, const void* base, int D, int64_t rows) {
  auto fn = dec_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kDecKeys)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int dec_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  return std::max(n, 1);
}

template <int D, int HG>
cudaError_t launch_dec(const DecodeArgs& a, const DecodeSplit& sp, cudaStream_t s) {
  const Problem& pr = a.p;
  const int64_t groups = static_cast<int64_t>(pr.B) * pr.Hkv;
  CUtensorMap tk, tv, tkd, tvd;
  if (!dec_map(&tk, a.k, D, groups * a.cap) || !dec_map(&tv, a.v, D, groups * a.cap)) return cudaErrorInvalidValue;
  if (pr.S > 0) {
    if (!dec_map(&tkd, a.kd, D, groups * pr.S) || !dec_map(&tvd, a.vd, D, groups * pr.S))
      return cudaErrorInvalidValue;
  } else {
    tkd = tk;
    tvd = tv;
  }
  DecParams p;
  p.B = pr.B;
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.T = pr.T;
  p.S = pr.S;
  p.S_read = pr.S_read;
  p.G = pr.G;
  p.n_seq = sp.n_seq;
  p.chunk = sp.chunk;
  p.cap = a.cap;
  p.scale_log2 = pr.scale_log2;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.part = a.part;
  p.status = a.status;
  using C = DecCfg<D>;
  static std::atomic<uint64_t> done{0};
  cudaError_t e = ensure_dynamic_smem(moda_decode_kernel<D, HG>, C::SMEM, done);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(sp.n_split), static_cast<unsigned>(groups));
  moda_decode_kernel<D, HG><<<grid, kDecThreads, C::SMEM, s>>>(tk, tv, tkd, tvd, p);
  DecMergeParams m;
  m.BH = pr.B * pr.H;
  m.n_split = sp.n_split;
  m.part = a.part;
  m.o = static_cast<__nv_bfloat16*>(a.o);
  m.lse = a.lse;
  moda_decode_merge_kernel<D><<<static_cast<unsigned>((m.BH + 3) / 4), 128, 0, s>>>(m);
  count_launches(2);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dec_d(const DecodeArgs& a, const DecodeSplit& sp, cudaStream_t s) {
  const int G = a.p.G;
  if (G == 1) return launch_dec<D, 1>(a, sp, s);
  if (G == 2) return launch_dec<D, 2>(a, sp, s);
  if (G <= 4) return launch_dec<D, 4>(a, sp, s);
  return launch_dec<D, 8>(a, sp, s);
}

}  // namespace

DecodeSplit decode_split(const Problem& p) {
  // About eight CTAs per SM, so that the last wave of equal-length splits leaves few SMs
  // idle, but at least 256 sequence keys per split.
  DecodeSplit sp;
  const int64_t groups = static_cast<int64_t>(p.B) * p.Hkv;
  const int by_keys = std::max(1, (p.T + 255) / 256);
  const int by_sms = static_cast<int>(std::max<int64_t>(1, (8 * dec_sms() + groups - 1) / groups));
  sp.n_seq = std::max(1, std::min({by_keys, by_sms, 1024}));
  const int per = (p.T + sp.n_seq - 1) / sp.n_seq;
  sp.chunk = (per + kDecKeys - 1) / kDecKeys * kDecKeys;
  sp.n_seq = (p.T + sp.chunk - 1) / sp.chunk;
  sp.n_split = sp.n_seq + (p.S > 0 ? 1 : 0);
  return sp;
}

bool decode_sm103_supported(const Problem& p) { return (p.d == 64 || p.d == 128) && p.G >= 1 && p.G <= kDecMaxG; }

cudaError_t launch_decode_sm103(const DecodeArgs& a, cudaStream_t s) {
  const DecodeSplit sp = decode_split(a.p);
  return a.p.d == 64 ? launch_dec_d<64>(a, sp, s) : launch_dec_d<128>(a, sp, s);
}

}  // namespace moda
