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
// G zero, into 16 TMEM columns), read back with lane = key; then lane = d/32 output
// columns for P V on the CUDA cores (P read back from shared memory as broadcasts).  Each warp keeps, per head, a running max,
// per-lane denominators and its output numerator; the CTA merges its warps and writes one
// partial state {max, sum, numerator} per head to a float32 workspace.  A second kernel
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

// Warps of a CTA: four key quarters for each head group.  One head group: splitting the
// heads over two groups of warps measured slower (both groups read and convert the same
// K and V rows).
template <int HG>
struct DecWarps {
  static constexpr int NHG = 1;        // head groups
  static constexpr int HS = HG / NHG;  // heads per group
  static constexpr int THREADS = 128 * NHG;
};

template <int D>
struct DecCfg {
  static constexpr int TILE_BYTES = kDecKeys * D * 2;  // one K (or V) sub-tile, bf16
  // One K slot and one V slot, each with a barrier of its own, and many resident CTAs
  // (three per SM at d = 128, six at d = 64): the other CTAs on the SM hide each one's
  // loads, and K of the next sub-tile loads while this one's softmax and P V run.
  static constexpr int OFF_K = 0, OFF_V = TILE_BYTES;
  // q of the heads as the B operand of the score product: bf16 [16 rows][D] (rows past G
  // zero), D/64 blocks of [16 rows x 128 B], 128-byte swizzle
  static constexpr int OFF_Q = 2 * TILE_BYTES;
  static constexpr int Q_BYTES = 16 * D * 2;
  // [4 warps][kDecMaxG][D + 2] float, used only after the last sub-tile has been read and
  // no copy is in flight: it shares the K/V slots
  static constexpr int OFF_RED = 0;
  static_assert(4 * kDecMaxG * (D + 2) * 4 <= 2 * TILE_BYTES, "reduction area");
  // float p [4 warps][32 keys][kDecMaxG]: the probabilities of each warp's keys, read back
  // as broadcasts in P V (one shared load per key instead of one shuffle per head)
  static constexpr int OFF_P = OFF_Q + Q_BYTES;
  static constexpr int OFF_BAR = OFF_P + 4 * 32 * kDecMaxG * 4;  // k_full, v_full, s_done, drain
  static constexpr int SMEM = OFF_BAR + 4 * 8 + 16;
  static constexpr uint32_t TM_COLS = 32;  // S^T: 128 lanes (keys) x 16 columns (heads)
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

__device__ __forceinline__ uint2 lds64v(uint32_t addr) {  // ordered after the preceding waits
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds32v(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Byte offset of 16-byte chunk x of row r in a [kDecKeys x D] bf16 tile stored as D/64
// blocks of [kDecKeys x 128 B], 128-byte swizzled (the layout TMA writes).
__device__ __forceinline__ uint32_t dec_off(int r, int x) {
  return static_cast<uint32_t>((x >> 3) * (kDecKeys * 128) + r * 128 + (((x & 7) ^ (r & 7)) << 4));
}

template <int D, int HG>
__global__ void __launch_bounds__(DecWarps<HG>::THREADS, 1)
    moda_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmKd, const __grid_constant__ CUtensorMap tmVd,
                       const DecParams p) {
  using C = DecCfg<D>;
  constexpr int CH = D / 8;    // 16-byte chunks per row
  constexpr int CPL = D / 32;  // output columns per lane
  constexpr int HS = DecWarps<HG>::HS;
  constexpr int NT = DecWarps<HG>::THREADS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kw = warp & 3, h0 = (warp >> 2) * HS;  // key quarter, first head of this warp
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

  // K of sub-tile s + 1 is loaded as soon as every warp has its scores for sub-tile s,
  // while the softmax and P V of s still run; V of s + 1 once P V of s is done
  uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* v_full = k_full + 1;
  uint64_t* s_done = k_full + 2;  // the score product of the current sub-tile is complete
  uint64_t* drain = k_full + 3;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 4 * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 4 * 8 + 4);
  float* pw = reinterpret_cast<float*>(smem + C::OFF_P) + kw * 32 * HS;  // this warp's [32][HS]
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    mbar_init(v_full, 1);
    mbar_init(s_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // q of the heads, bf16, rows past G zero: 16-byte chunk x of row hh
  for (int i = threadIdx.x; i < 16 * CH; i += NT) {
    const int hh = i / CH, x = i % CH;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (hh < p.G) v = *reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(b) * p.H + g * p.G + hh) * D + x * 8);
    st_shared_v4(sbase + C::OFF_Q + (x >> 3) * (16 * 128) + hh * 128 + (((x & 7) ^ (hh & 7)) << 4), v);
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the score product: A = the K sub-tile (keys x D, K-major), B = q (16 rows x D, K-major)
  constexpr uint32_t IDESC_S = idesc_bf16(kDecKeys, 16, false);
  const uint64_t a_desc = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
  const uint64_t b_desc = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
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

  float m[HS], l[HS], o[HS][CPL];
#pragma unroll
  for (int hh = 0; hh < HS; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[hh][c] = 0.f;
  }
  const int r = kw * 32 + lane;  // this lane's key row within a sub-tile
  int issued_k = min(n_sub, 1), issued_v = issued_k;  // sub-tiles whose K / V loads are issued
  bool failed = false;
  int mma_issued = 0;  // score products issued (thread 0)
  for (int s = 0; s < n_sub; ++s) {
    const uint32_t par = s & 1;
    if (__syncthreads_or(!mbar_wait(k_full, par, abort_flag))) {  // block-uniform
      failed = true;
      break;
    }
    const uint32_t vt = sbase + C::OFF_V;
    const int base_key = s * kDecKeys;
    // ---- scores of the heads for the sub-tile's keys on the tensor core
    if (threadIdx.x == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16_ss(tmem, sdesc_add(a_desc, (kk >> 2) * (kDecKeys * 128) + (kk & 3) * 32),
                    sdesc_add(b_desc, (kk >> 2) * (16 * 128) + (kk & 3) * 32), IDESC_S, kk > 0);
      mma_commit(s_done);
      ++mma_issued;
    }
    if (__syncthreads_or(!mbar_wait(s_done, par, abort_flag))) {
      failed = true;
      break;
    }
    tc_fence_after();
    uint32_t sv[16];
    tmem_ld16(tmem + (static_cast<uint32_t>(kw * 32) << 16), sv);  // lane = key r, column = head
    tc_fence_before();
    // every warp has its scores (the product has read K): load the next sub-tile's K
    __syncthreads();
    if (threadIdx.x == 0 && issued_k < n_sub) issue(issued_k, 0);
    ++issued_k;
    const bool valid = base_key + r < n_keys;
    // ---- online softmax per head: warp-wide max, per-lane sums
    float pr[HS], sc[HS], wmax[HS];
#pragma unroll
    for (int hh = 0; hh < HS; ++hh) sc[hh] = valid ? __uint_as_float(sv[h0 + hh]) * p.scale_log2 : -INFINITY;
    if constexpr (HS == 4) {
      // reduce-scatter of the four maxima over lane bits 4 and 3, a butterfly over bits
      // 2..0, then a gather: 10 shuffles instead of 20 (a shuffle issues at a quarter of
      // the FMA rate)
      const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0;
      float y[2];
#pragma unroll
      for (int u = 0; u < 2; ++u)
        y[u] = fmaxf(b4 ? sc[u + 2] : sc[u], __shfl_xor_sync(0xffffffffu, b4 ? sc[u] : sc[u + 2], 16));
      float z = fmaxf(b3 ? y[1] : y[0], __shfl_xor_sync(0xffffffffu, b3 ? y[0] : y[1], 8));
#pragma unroll
      for (int off = 4; off >= 1; off >>= 1) z = fmaxf(z, __shfl_xor_sync(0xffffffffu, z, off));
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) wmax[hh] = __shfl_sync(0xffffffffu, z, hh * 8);  // lane of head hh
    } else {
#pragma unroll
      for (int hh = 0; hh < HS; ++hh) {
        float wm = sc[hh];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, off));
        wmax[hh] = wm;
      }
    }
#pragma unroll
    for (int hh = 0; hh < HS; ++hh) {
      const float m_new = fmaxf(m[hh], wmax[hh]);
      const float corr = (m[hh] == -INFINITY) ? 0.f : ex2(m[hh] - m_new);
      pr[hh] = valid ? ex2(sc[hh] - m_new) : 0.f;
      l[hh] = l[hh] * corr + pr[hh];
#pragma unroll
      for (int c = 0; c < CPL; ++c) o[hh][c] *= corr;
      m[hh] = m_new;
    }
    if (__syncthreads_or(!mbar_wait(v_full, par, abort_flag))) {
      failed = true;
      break;
    }
    // this lane's probabilities for the warp's P V loop (the previous sub-tile's loop has
    // read its values before the barriers above)
#pragma unroll
    for (int hh = 0; hh < HS; ++hh) pw[lane * HS + hh] = pr[hh];
    __syncwarp();
    // ---- P V over this warp's valid keys; lane owns columns [lane*CPL, lane*CPL + CPL)
    const int n_here = min(32, n_keys - base_key - kw * 32);  // warp-uniform
    const int xc = (lane * CPL) >> 3, sub = ((lane * CPL) & 7) * 2;
    for (int j = 0; j < n_here; ++j) {
      const int rv = kw * 32 + j;
      float vf[CPL];
      if constexpr (CPL == 4) {
        const uint2 vw = lds64v(vt + dec_off(rv, xc) + sub);
        vf[0] = bf16_lo(vw.x);
        vf[1] = bf16_hi(vw.x);
        vf[2] = bf16_lo(vw.y);
        vf[3] = bf16_hi(vw.y);
      } else {
        const uint32_t vw = lds32v(vt + dec_off(rv, xc) + sub);
        vf[0] = bf16_lo(vw);
        vf[1] = bf16_hi(vw);
      }
#pragma unroll
      for (int hh = 0; hh < HS; ++hh) {
        const float pj = pw[j * HS + hh];
#pragma unroll
        for (int c = 0; c < CPL; c += 2) ffma2(pj, pj, vf[c], vf[c + 1], o[hh][c], o[hh][c + 1], o[hh][c], o[hh][c + 1]);
      }
    }
    // every warp has read V: load the next sub-tile's V
    __syncthreads();
    if (threadIdx.x == 0 && issued_v < n_sub) issue(issued_v, 1);
    ++issued_v;
  }
  if (failed) {
    if (threadIdx.x == 0) {
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
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TM_COLS);
    }
    return;
  }
  // every score product has been read (the s_done waits): TMEM is no longer needed
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
  // ---- merge the four key-quarter warps' states of each head into this split's state
#pragma unroll
  for (int hh = 0; hh < HS; ++hh) {
    float ls = l[hh];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
    float* w = red + (kw * kDecMaxG + h0 + hh) * (D + 2);
    if (lane == 0) {
      w[0] = m[hh];
      w[1] = ls;
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) w[2 + lane * CPL + c] = o[hh][c];
  }
  __syncthreads();
  const int64_t row_base = static_cast<int64_t>(split) * p.B * p.H + static_cast<int64_t>(b) * p.H + g * p.G;
  for (int i = threadIdx.x; i < p.G * (D + 2); i += NT) {
    const int hh = i / (D + 2), e = i % (D + 2);
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) mx = fmaxf(mx, red[(w * kDecMaxG + hh) * (D + 2)]);
    float val;
    if (e == 0) {
      val = mx;
    } else {
      val = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = red[(w * kDecMaxG + hh) * (D + 2)];
        if (mw != -INFINITY) val += red[(w * kDecMaxG + hh) * (D + 2) + e] * ex2(mw - mx);
      }
    }
    p.part[(row_base + hh) * (D + 2) + e] = val;
  }
}

struct DecMergeParams {
  int BH, n_split;
  const float* part;
  __nv_bfloat16* o;
  float* lse;  // may be null
};

// One warp per (b, h): merge the splits' partial states by the online rule, divide once.
template <int D>
__global__ void __launch_bounds__(128) moda_decode_merge_kernel(const DecMergeParams p) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= p.BH) return;
  float mx = -INFINITY;
  for (int s = 0; s < p.n_split; ++s) mx = fmaxf(mx, p.part[(static_cast<int64_t>(s) * p.BH + row) * (D + 2)]);
  float L = 0.f, acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
  for (int s = 0; s < p.n_split; ++s) {
    const float* ps = p.part + (static_cast<int64_t>(s) * p.BH + row) * (D + 2);
    const float ms = ps[0];
    if (ms == -INFINITY) continue;  // a split without keys
    const float w = ex2(ms - mx);
    L += ps[1] * w;
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
  moda_decode_kernel<D, HG><<<grid, DecWarps<HG>::THREADS, C::SMEM, s>>>(tk, tv, tkd, tvd, p);
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
