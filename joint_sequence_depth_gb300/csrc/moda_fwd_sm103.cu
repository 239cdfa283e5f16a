// MoDA forward on the sm_103a tensor cores: tcgen05 MMAs into TMEM fed by TMA,
// with the same-position depth slots folded in on the CUDA cores.
//
// Operation: "Mixture-of-Depths Attention", frame "One denominator allocates
// probability across both memories" (Sec. 2.2, Algorithm 1): one softmax over
// the causal sequence keys and the depth slots of the query's own position.
//
// Tile.  A CTA owns 128 expanded query rows of one (batch b, kv head g): the
// G query heads of g at P = floor(128/G) consecutive positions, row r ->
// (position p0 + r/G, head g*G + r%G).  This is the grouped row expansion of
// frame "Backup: grouped indexing preserves the correct token map" (T_q = G*T_kv,
// t_base = floor(i_q/G)): every K/V tile of kv head g is loaded once for all G
// heads, and the [S, d] depth slab of a position is read once for its G rows
// (the group-aware reuse of Sec. 3.2 / Fig. 4, without its packed layout).
//
// Warp roles (384 threads):
//   warp 0      TMA producer: K_j, V_j tiles of 128 keys into a ring of smem slots.
//   warp 1      TMEM allocator and MMA issuer (one thread):
//                 S_j = Q K_j^T   (M=128, N=128, K=d), A and B from smem, into TMEM S[j%2]
//                 O  += P_j V_j   (M=128, N=d,  K=128), A = P_j from TMEM, B from smem
//   warp 2      depth producer: bulk copies of each position's [SC, d] depth sub-slabs
//               (K then V, SC slots at a time) into one smem ring per depth warp, the
//               slabs of neighbouring positions staggered by 16 bytes so the depth
//               warps' 128-bit shared loads do not collide on banks.
//   warps 4-7   softmax: thread r owns row r (TMEM lane r); online softmax over S_j
//               with running max m and denominator l (frame "Shared online-softmax
//               states preserve the joint operator"), exp2 with a log2(e)-folded
//               scale; P_j rounded to bf16 and written back into the TMEM columns of
//               S_j; O rescaled in TMEM only when the running max grows by more than
//               2^8 (exact: the final division uses the same stale max); epilogue.
//   warps 8-11  Q loader + depth: thread r loads row r of Q (registers and smem for
//               the MMAs), then folds the S depth slots of its position SC at a time:
//               scores with bf16 x bf16 -> fp32 FMAs, the same online update
//               (m_d, l_d), and o_d accumulated in TMEM columns Od.
// The epilogue merges the two running states with the online-softmax update rule
// and divides once: o = (e^{m_s-m} O + e^{m_d-m} Od) / (e^{m_s-m} l_s + e^{m_d-m} l_d),
// the single denominator of the joint operator.
//
// TMEM columns: S0 [0,128), S1 [128,256), O [256,256+d), Od [256+d,256+2d); P_j is
// packed bf16 in the first 64 columns of S[j%2].
#include <cudaTypedefs.h>

#include <algorithm>

#include "moda_common.cuh"
#include "sm103_ptx.cuh"

namespace moda {
namespace {

using namespace sm103;

constexpr int BM = 128;                    // expanded query rows per CTA
constexpr int BN = 128;                    // keys per K/V tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kDepthWarps = 4;
constexpr int kDepthStages = 2;
constexpr int kSmemLimit = 232448;  // bytes of dynamic shared memory a CTA may use

// Shared memory: Q tile | K/V ring (NSLOT tiles) | depth rings (4 warps x 2 stages of
// `dstage` bytes, sized on the host) | barriers | misc.  With NSLOT >= 4 the load of
// K_{j+2} only waits for K_j's slot, so it is in flight while PV_j runs.
template <int D, int SC, int NSLOT_>
struct FwdCfg {
  static constexpr int NSLOT = NSLOT_;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int SUB = SC * D * 2;   // one position's sub-slab of SC slots
  static constexpr int STRIDE = SUB + 16;  // staggered position stride in a stage
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + Q_BYTES;
  static constexpr int OFF_DEP = OFF_KV + NSLOT * KV_BYTES;
  // kv_full[NSLOT], kv_empty[NSLOT], q_full, s_full[2], p_full[2], pv_done[2], depth_done, drain,
  // dfull[4*NB], dempty[4*NB]
  static constexpr int NBAR = 2 * NSLOT + 9 + 2 * kDepthWarps * kDepthStages;
  static constexpr int TAIL = NBAR * 8 + 16 + 2 * BM * 4;  // barriers, misc words, m_d[], l_d[]
  static constexpr uint32_t TM_S0 = 0, TM_O = 256, TM_OD = 256 + D;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int off_bar(int dstage) { return OFF_DEP + kDepthWarps * kDepthStages * dstage; }
  static constexpr int smem_alloc(int dstage) { return off_bar(dstage) + TAIL; }
};

struct FwdTcParams {
  int B, H, Hkv, T, S, G, P, n_pb;
  int dstage;  // bytes of one depth ring stage (multiple of 16)
  float scale_log2;
  const __nv_bfloat16* q;
  const __nv_bfloat16* kd;
  const __nv_bfloat16* vd;
  __nv_bfloat16* o;
  float* lse;
  int* status;
};

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  record_status(status, kStatusTimeout);
}

// All lanes wait on the same barrier phase; the warp takes one decision.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

template <int D, int SC, int NSLOT>
__global__ void __launch_bounds__(384, 1)
    moda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const FwdTcParams p) {
  using C = FwdCfg<D, SC, NSLOT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  // The 128-byte swizzle atoms need 1024-byte aligned tiles; the dynamic shared window
  // starts 1024-aligned on this architecture, and a launch where it does not is refused.
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = p.B * p.Hkv;
  const int pb = p.n_pb - 1 - static_cast<int>(blockIdx.x) / ngroups;  // heaviest position blocks first
  const int bg = static_cast<int>(blockIdx.x) % ngroups;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int p0 = pb * p.P;
  const int p_last = min(p0 + p.P, p.T) - 1;
  const int n_kv = p_last / BN + 1;
  const int n_dchunks = (p.S + SC - 1) / SC;  // depth slot groups (each: K pass then V pass)

  const int off_bar = C::off_bar(p.dstage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + off_bar);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::NSLOT;
  uint64_t* q_full = bars + 2 * C::NSLOT;
  uint64_t* s_full = q_full + 1;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* depth_done = pv_done + 2;
  uint64_t* drain = depth_done + 1;
  uint64_t* dfull = drain + 1;
  uint64_t* dempty = dfull + kDepthWarps * kDepthStages;
  uint8_t* misc = smem + off_bar + C::NBAR * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  float* md_s = reinterpret_cast<float*>(misc + 16);
  float* ld_s = md_s + BM;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(q_full, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(depth_done, 128);
    mbar_init(drain, 1);
    for (int i = 0; i < kDepthWarps * kDepthStages; ++i) {
      mbar_init(&dfull[i], 1);
      mbar_init(&dempty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (K/V)
    if (lane == 0) {
      const int n_items = 2 * n_kv;  // K0, V0, K1, V1, ...
      int issued = 0;
      for (int it = 0; it < n_items; ++it) {
        const int slot = it % C::NSLOT, use = it / C::NSLOT;
        if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, abort_flag)) {
          raise_abort(abort_flag, p.status);
          break;
        }
        const int j = it >> 1;
        const CUtensorMap* map = (it & 1) ? &tmV : &tmK;
        uint8_t* dst = smem + C::OFF_KV + slot * C::KV_BYTES;
        mbar_arrive_expect_tx(&kv_full[slot], C::KV_BYTES);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * (BN * 128), map, &kv_full[slot], h * 64, j * BN, bg);
        issued = it + 1;
      }
      if (*abort_flag) {
        // let every copy still in flight land before the CTA exits
        volatile int never = 0;
        for (int it = max(0, issued - C::NSLOT); it < issued; ++it)
          mbar_wait(&kv_full[it % C::NSLOT], (it / C::NSLOT) & 1, &never);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false);
      constexpr uint32_t IDESC_O = idesc_bf16(BM, D, true);
      // descriptors built once; each MMA only advances the start address
      const uint64_t q_desc = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t kv_desc_k = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);          // K-major (K tiles)
      const uint64_t kv_desc_v = sdesc_sw128(sbase + C::OFF_KV, BN * 128, 1024);    // MN-major (V tiles)
      bool ok = mbar_wait(q_full, 0, abort_flag);
      auto issue_s = [&](int j) -> bool {
        const int it = 2 * j, slot = it % C::NSLOT;
        if (!mbar_wait(&kv_full[slot], (it / C::NSLOT) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t k_desc = sdesc_add(kv_desc_k, slot * C::KV_BYTES);
        const uint32_t d_tmem = tmem + C::TM_S0 + (j & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          mma_bf16_ss(d_tmem, sdesc_add(q_desc, (kk >> 2) * (BM * 128) + (kk & 3) * 32),
                      sdesc_add(k_desc, (kk >> 2) * (BN * 128) + (kk & 3) * 32), IDESC_S, kk > 0);
        }
        mma_commit(&s_full[j & 1]);
        mma_commit(&kv_empty[slot]);
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag)) return false;
        const int it = 2 * j + 1, slot = it % C::NSLOT;
        if (!mbar_wait(&kv_full[slot], (it / C::NSLOT) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t p_tmem = tmem + C::TM_S0 + (j & 1) * BN;
        const uint64_t v_desc = sdesc_add(kv_desc_v, slot * C::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          mma_bf16_ts(tmem + C::TM_O, p_tmem + kk * 8, sdesc_add(v_desc, kk * 16 * 128), IDESC_O,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&pv_done[j & 1]);
        mma_commit(&kv_empty[slot]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n_kv > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n_kv; ++j) {
        ok = issue_pv(j);
        if (ok && j + 2 < n_kv) ok = issue_s(j + 2);
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        // wait for every MMA already issued before TMEM is released
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- depth producer
    // Chunk c = 2*cs + kind (kind 0: Kd, 1: Vd) holds slots [cs*SC, cs*SC+SC) of every
    // position of a consumer warp, one bulk copy per position (lane = position).
    bool ok = true;
    int c = 0, w = 0;
    for (c = 0; ok && c < 2 * n_dchunks; ++c) {
      const int i0 = (c >> 1) * SC, nc = min(SC, p.S - i0);
      const int stage = c % kDepthStages, use = c / kDepthStages;
      const __nv_bfloat16* src_base = (c & 1) ? p.vd : p.kd;
      for (w = 0; w < kDepthWarps; ++w) {
        const int bi = w * kDepthStages + stage;
        if (use > 0 && !warp_wait(&dempty[bi], (use - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int kw0 = (32 * w) / p.G;
        const int kw1 = min((32 * w + 31) / p.G, min(p.P, p.T - p0) - 1);
        const int nvalid = max(0, kw1 - kw0 + 1);
        const uint32_t bytes = static_cast<uint32_t>(nc) * D * 2;
        if (lane == 0) mbar_arrive_expect_tx(&dfull[bi], bytes * nvalid);
        __syncwarp();
        if (lane < nvalid) {
          const int k = kw0 + lane;
          const __nv_bfloat16* src = src_base + ((static_cast<int64_t>(bg) * p.T + p0 + k) * p.S + i0) * D;
          const uint32_t dst = sbase + C::OFF_DEP + bi * p.dstage + lane * C::STRIDE;
          bulk_load(dst, src, bytes, &dfull[bi]);
        }
      }
      if (!ok) break;
    }
    if (!ok) {
      if (lane == 0) raise_abort(abort_flag, p.status);
      // Copies possibly in flight: every warp's share of the chunks after the last stage
      // reuse, and warps < w of chunk c.  Let them land before the CTA exits.
      volatile int never = 0;
      for (int cc = max(0, c - kDepthStages + 1); cc <= c; ++cc)
        for (int ww = 0; ww < kDepthWarps && (cc < c || ww < w); ++ww)
          mbar_wait(&dfull[ww * kDepthStages + cc % kDepthStages], (cc / kDepthStages) & 1, &never);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------------- softmax
    const int r = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int pos = p0 + r / p.G;
    const bool valid = (r < p.P * p.G) && pos < p.T;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = warp_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_tmem = tmem + lane_base + C::TM_S0 + (j & 1) * BN;
      uint32_t s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_tmem + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
      const int kb = j * BN;
      if (kb + BN - 1 > p0 || !valid) {
        // diagonal tile (or dead row): keys after the row's position are invisible
        const int lim = valid ? pos - kb : -1;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c > lim) s[c] = __float_as_uint(-INFINITY);
      }
      // row max: four independent chains of 3-input max
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; c += 8) {
        mx0 = fmax3(mx0, __uint_as_float(s[c + 0]), __uint_as_float(s[c + 1]));
        mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
        mx2 = fmax3(mx2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
        mx3 = fmax3(mx3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
      }
      const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
      if (j == 0) {
        m_run = m_tile;
      } else {
        const bool need = m_tile > m_run + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_run, m_tile);
          const float corr = (m_run == -INFINITY) ? 1.f : ex2(m_run - m_new);
          // PV_{j-1} must have landed in O before it is rescaled
          ok = warp_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + C::TM_O + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tmem_st32(tmem + lane_base + C::TM_O + c * 32, o);
          }
          l_run *= corr;
          m_run = m_new;
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // p = 2^(s*scale*log2e - m): packed FMA, MUFU ex2, packed row-sum in four chains
      float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN; c += 4) {
        float x0, x1, x2, x3;
        ffma2_bc(__uint_as_float(s[c]), __uint_as_float(s[c + 1]), sl2, -m_use, x0, x1);
        ffma2_bc(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]), sl2, -m_use, x2, x3);
        x0 = ex2(x0);
        x1 = ex2(x1);
        x2 = ex2(x2);
        x3 = ex2(x3);
        if ((c & 4) == 0)
          fadd2(ls0, ls1, x0, x1), fadd2(ls0, ls1, x2, x3);
        else
          fadd2(ls2, ls3, x0, x1), fadd2(ls2, ls3, x2, x3);
        pk[c >> 1] = pack_bf16(x0, x1);
        pk[(c >> 1) + 1] = pack_bf16(x2, x3);
      }
      l_run += (ls0 + ls1) + (ls2 + ls3);
      // P_j (bf16 pairs) into the first 64 columns of S_j's TMEM buffer
      tmem_st32(s_tmem, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(s_tmem + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }
    if (!ok) {
      raise_abort(abort_flag, p.status);
    } else {
      // ------------------------------------------------------------ epilogue
      const int jl = n_kv - 1;
      ok = warp_wait(&pv_done[jl & 1], (jl >> 1) & 1, abort_flag) && warp_wait(depth_done, 0, abort_flag);
      if (!ok) {
        raise_abort(abort_flag, p.status);
      } else {
        tc_fence_after();
        const float md = md_s[r], ldp = ld_s[r];
        const float m = fmaxf(m_run, md);
        const float a_s = (l_run > 0.f) ? ex2(m_run - m) : 0.f;
        const float a_d = (ldp > 0.f) ? ex2(md - m) : 0.f;
        const float L = l_run * a_s + ldp * a_d;
        const float inv = valid ? 1.f / L : 0.f;
        const float ws = a_s * inv, wd = a_d * inv;
        const int h = g * p.G + r % p.G;
        __nv_bfloat16* orow = p.o + ((static_cast<int64_t>(b) * p.H + h) * p.T + (valid ? pos : 0)) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t os[32], od[32];
          tmem_ld32(tmem + lane_base + C::TM_O + c * 32, os);
          if (p.S > 0) {
            tmem_ld32(tmem + lane_base + C::TM_OD + c * 32, od);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) od[i] = 0u;
          }
          uint32_t pk2[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float x0 = __uint_as_float(os[i]) * ws + __uint_as_float(od[i]) * wd;
            const float x1 = __uint_as_float(os[i + 1]) * ws + __uint_as_float(od[i + 1]) * wd;
            pk2[i >> 1] = pack_bf16(x0, x1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk2[4 * i], pk2[4 * i + 1], pk2[4 * i + 2], pk2[4 * i + 3]);
          }
        }
        if (valid && p.lse != nullptr)
          p.lse[(static_cast<int64_t>(b) * p.H + h) * p.T + pos] = (m + __log2f(L)) * kLn2;
      }
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------------------- Q loader + depth
    const int w = warp - 8;
    const int r = threadIdx.x - 256;
    const uint32_t lane_base = static_cast<uint32_t>(w * 32) << 16;
    const int k = r / p.G;
    const int pos = p0 + k;
    const bool valid = (r < p.P * p.G) && pos < p.T;
    const int h = g * p.G + r % p.G;
    const uint32_t q_base = sbase + C::OFF_Q;
    uint4 qv[D / 8];
    {
      const uint4* qrow =
          reinterpret_cast<const uint4*>(p.q + ((static_cast<int64_t>(b) * p.H + h) * p.T + (valid ? pos : 0)) * D);
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {
        qv[ch] = valid ? __ldg(qrow + ch) : make_uint4(0u, 0u, 0u, 0u);
        st_shared_v4(q_base + (ch >> 3) * (BM * 128) + sw128_offset(r, ch & 7), qv[ch]);
      }
      fence_proxy_async_smem();
      mbar_arrive(q_full);
    }
    float m_d = -INFINITY, l_d = 0.f;
    bool ok = true;
    const int kl = k - (32 * w) / p.G;  // position index inside this warp's stage layout
    const float sl2 = p.scale_log2;
    for (int cs = 0; cs < n_dchunks; ++cs) {
      const int i0 = cs * SC, nc = min(SC, p.S - i0);
      // ---- K pass: scores of slots [i0, i0+nc)
      int c = 2 * cs;
      int bi = w * kDepthStages + c % kDepthStages;
      ok = warp_wait(&dfull[bi], (c / kDepthStages) & 1, abort_flag);
      if (!ok) break;
      // two partial sums per slot (even / odd 16-byte chunks) for instruction-level parallelism
      float sc[SC], sc2[SC];
#pragma unroll
      for (int i = 0; i < SC; ++i) sc[i] = sc2[i] = 0.f;
      if (valid) {
        const uint32_t kbuf = sbase + C::OFF_DEP + bi * p.dstage + kl * C::STRIDE;
#pragma unroll
        for (int ch = 0; ch < D / 8; ++ch) {
#pragma unroll
          for (int i = 0; i < SC; ++i) {
            if (i < nc) {
              const uint4 kv = ld_shared_v4(kbuf + i * (D * 2) + ch * 16);
              float a = (ch & 1) ? sc2[i] : sc[i];
              a = dot2_bf16(qv[ch].x, kv.x, a);
              a = dot2_bf16(qv[ch].y, kv.y, a);
              a = dot2_bf16(qv[ch].z, kv.z, a);
              a = dot2_bf16(qv[ch].w, kv.w, a);
              if (ch & 1)
                sc2[i] = a;
              else
                sc[i] = a;
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < SC; ++i) sc[i] += sc2[i];
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[bi]);
      // ---- online update of (m_d, l_d) with this slot group
      float cmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < SC; ++i)
        if (i < nc && valid) cmax = fmaxf(cmax, sc[i] * sl2);
      const float m_new = fmaxf(m_d, cmax);
      const float corr = (m_d == -INFINITY) ? 0.f : ex2(m_d - m_new);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      uint32_t pb[SC];
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < SC; ++i) {
        const float e = (i < nc && valid) ? ex2(fmaf(sc[i], sl2, -m_use)) : 0.f;
        psum += e;
        pb[i] = pack_bf16(e, 0.f);
      }
      l_d = l_d * corr + psum;
      // ---- V pass: o_d = corr * o_d + sum_i p_i vd_i, accumulated in TMEM Od
      c = 2 * cs + 1;
      bi = w * kDepthStages + c % kDepthStages;
      ok = warp_wait(&dfull[bi], (c / kDepthStages) & 1, abort_flag);
      if (!ok) break;
      const uint32_t vbuf = sbase + C::OFF_DEP + bi * p.dstage + kl * C::STRIDE;
#pragma unroll 1
      for (int g32 = 0; g32 < D / 32; ++g32) {
        uint32_t acc[32];
        if (cs == 0) {
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0u;
        } else {
          tmem_ld32(tmem + lane_base + C::TM_OD + g32 * 32, acc);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = __float_as_uint(__uint_as_float(acc[i]) * corr);
        }
        if (valid) {
          float* a = reinterpret_cast<float*>(acc);
#pragma unroll
          for (int i = 0; i < SC; ++i) {
            if (i < nc) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                const uint4 vv = ld_shared_v4(vbuf + i * (D * 2) + (g32 * 4 + q4) * 16);
                axpy2_bf16(pb[i], vv.x, a[8 * q4 + 0], a[8 * q4 + 1]);
                axpy2_bf16(pb[i], vv.y, a[8 * q4 + 2], a[8 * q4 + 3]);
                axpy2_bf16(pb[i], vv.z, a[8 * q4 + 4], a[8 * q4 + 5]);
                axpy2_bf16(pb[i], vv.w, a[8 * q4 + 6], a[8 * q4 + 7]);
              }
            }
          }
        }
        tmem_st32(tmem + lane_base + C::TM_OD + g32 * 32, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[bi]);
      m_d = m_new;
    }
    if (!ok) raise_abort(abort_flag, p.status);
    md_s[r] = m_d;
    ld_s[r] = l_d;
    tc_fence_before();
    mbar_arrive(depth_done);
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// [groups = B*Hkv][T][D] bf16 viewed as a 3-D tensor (D, T, groups); box 64 x 128 x 1,
// 128-byte swizzle; rows past T read as zeros.
bool make_kv_map(CUtensorMap* map, const void* base, int D, int T, int groups) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(groups)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BN), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Most positions any depth warp covers (its 32 rows of the position-major tile).
int positions_per_warp(int G, int P) {
  int most = 0;
  for (int w = 0; w < kDepthWarps; ++w) {
    const int k0 = (32 * w) / G, k1 = std::min((32 * w + 31) / G, P - 1);
    most = std::max(most, k1 - k0 + 1);
  }
  return most;
}

// Depth stage bytes for slot groups of SC: the staggered sub-slabs of the most positions
// one depth warp covers.
int depth_stage_bytes(int npos, int sc, int D) { return npos * (sc * D * 2 + 16); }

template <int D, int SC, int NSLOT>
bool fits(int npos) {
  return FwdCfg<D, SC, NSLOT>::smem_alloc(depth_stage_bytes(npos, SC, D)) <= kSmemLimit;
}

template <int D, int SC, int NSLOT>
cudaError_t launch_cfg(FwdTcParams p, int npos, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
  using C = FwdCfg<D, SC, NSLOT>;
  p.dstage = depth_stage_bytes(npos, SC, D);
  const int smem = C::smem_alloc(p.dstage);
  static int attr_bytes = 0;
  if (attr_bytes < smem) {
    cudaError_t e =
        cudaFuncSetAttribute(moda_fwd_tc_kernel<D, SC, NSLOT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_bytes = smem;
  }
  const unsigned grid = static_cast<unsigned>(p.n_pb) * p.B * p.Hkv;
  moda_fwd_tc_kernel<D, SC, NSLOT><<<grid, 384, smem, s>>>(tk, tv, p);
  count_launches(1);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch(const FwdArgs& a, cudaStream_t s) {
  const Problem& pr = a.p;
  CUtensorMap tk, tv;
  if (!make_kv_map(&tk, a.k, D, pr.T, pr.B * pr.Hkv) || !make_kv_map(&tv, a.v, D, pr.T, pr.B * pr.Hkv))
    return cudaErrorInvalidValue;
  FwdTcParams p;
  p.B = pr.B;
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.T = pr.T;
  p.S = pr.S;
  p.G = pr.G;
  p.P = BM / pr.G;
  p.n_pb = (pr.T + p.P - 1) / p.P;
  p.scale_log2 = pr.scale_log2;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kd = static_cast<const __nv_bfloat16*>(a.kd);
  p.vd = static_cast<const __nv_bfloat16*>(a.vd);
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.status = a.status;
  // Prefer a 4-deep K/V ring (6-deep at d=64), then the largest depth slot group that fits.
  const int npos = positions_per_warp(pr.G, p.P);
  constexpr int NS = D == 128 ? 4 : 6;
  if (fits<D, 8, NS>(npos)) return launch_cfg<D, 8, NS>(p, npos, tk, tv, s);
  if (fits<D, 4, NS>(npos)) return launch_cfg<D, 4, NS>(p, npos, tk, tv, s);
  if (fits<D, 2, NS>(npos)) return launch_cfg<D, 2, NS>(p, npos, tk, tv, s);
  if (fits<D, 1, NS>(npos)) return launch_cfg<D, 1, NS>(p, npos, tk, tv, s);
  if (fits<D, 2, NS - 1>(npos)) return launch_cfg<D, 2, NS - 1>(p, npos, tk, tv, s);
  return launch_cfg<D, 1, NS - 1>(p, npos, tk, tv, s);
}

}  // namespace

bool fwd_sm103_supported(const Problem& p) { return (p.d == 64 || p.d == 128) && p.G >= 1 && p.G <= BM; }

cudaError_t launch_fwd_sm103(const FwdArgs& a, cudaStream_t s) {
  return a.p.d == 64 ? launch<64>(a, s) : launch<128>(a, s);
}

}  // namespace moda
