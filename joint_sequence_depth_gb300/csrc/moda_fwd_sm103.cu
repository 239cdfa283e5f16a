// MoDA forward on the sm_103a tensor cores: a persistent kernel with two ping-pong
// query tiles per work unit and tcgen05 MMAs into TMEM fed by TMA, in which the
// same-position depth slots of all the tile's positions enter as one extra key step.
//
// Operation: "Mixture-of-Depths Attention", frame "One denominator allocates
// probability across both memories" (Sec. 2.2, Algorithm 1): one softmax over the
// causal sequence keys and the depth slots of the query's own position.
//
// Work unit.  256 expanded query rows of one (batch b, kv head g): two tiles of 128
// rows, tile t holding the G query heads of g at the P = floor(128/G) positions
// p0 + t*P .. p0 + t*P + P - 1, position-major: row r -> (position p0 + t*P + r/G,
// head g*G + r%G), the grouped row expansion of frame "Backup: grouped indexing
// preserves the correct token map" (T_q = G*T_kv).  One 4-D TMA box per 64 columns
// loads a tile: Q [B][H][T][d] is described to the TMA unit as (d, H, T, B), so the
// box walks the G heads fastest.
//
// Key steps of a query tile t, in the order the online softmax takes them:
//   depth steps i = 0 .. n_d-1 (n_d = ceil(S_read / 128), one unless more than 128 slots
//     are read).  The read slots 128 i .. 128 i + w - 1 (w = min(S_read, 128)) of the
//     tile's positions come in chunks of dpt = floor(128 / w) positions, one 3-D TMA box
//     (channels, slots, positions) each: key kappa of chunk c is slot 128 i + kappa % w of
//     local position c*dpt + kappa / w (slots past S_read read as zeros; slots never read
//     are never loaded).  Chunk c's S = Q K_c^T and O += P V_c are tensor-core products
//     over all 128 rows whose TMEM write-back is masked to the rows of the chunk's
//     positions (the disable-output-lane operand), so every chunk writes the same S and
//     reads the same P columns and the step's softmax covers all chunks at once: row r
//     sees columns [(r/G - c*dpt) w, + w) of its own chunk's keys.  This is the
//     same-position depth memory H_l of the slides' formulas, scored by the same MMAs as
//     the sequence.
//   sequence steps j = 0 .. : keys 128 j .. 128 j + 127 of kv head g, causal mask: key
//               j is visible to position t when j <= t + delta and j < Tk.  A whole
//               sequence has delta = 0 and Tk = T; a query chunk scored against the key
//               chunk of an earlier range of positions (context parallelism) has the
//               offset delta = (first query position) - (first key position) > 0.
// Both kinds go through the same running max m and denominator l, the shared
// online-softmax state of frame "Shared online-softmax states preserve the joint
// operator", and one PV accumulator O: the depth slots are never normalised apart.
// Each K/V tile of the sequence is loaded once for the G heads and both query tiles,
// each depth slab once for its G rows (the group-aware reuse of Sec. 3.2 / Fig. 4).
//
// Units are ordered heaviest first and dealt to the persistent CTAs in a snake order.
//
// Warp roles (384 threads):
//   warp 0      TMA: the two Q tiles of each unit, then the K/V items of the unit in the
//               order the MMA warps consume them, into a ring of smem slots.
//   warp 1      TMEM allocator.  d = 128: the MMA-issuing warp for both tiles.  Per step i:
//                 PV_0(i), S_0(i+1), PV_1(i), S_1(i+1)  with  S_t = Q_t K^T into TMEM
//                 S[t] and O_t += P_t V (P_t read from TMEM), so the tensor core works on
//                 one tile while the other tile's softmax runs.
//   warps 1, 2  d = 64: one MMA-issuing warp per query tile; S_t of the next key tile is
//               issued as soon as the softmax warps have read S_t (P_t has columns of its
//               own), so S and the softmax overlap within a tile as well.
//               The issuing warps run their loops warp-wide (every lane takes the waits
//               and the decisions) and one elected lane issues each MMA group: a loop run
//               by lane 0 alone issues markedly slower while softmax warps keep the SM
//               sub-partition busy (measured on GB300: 79-89 against 64 cycles per
//               128x128x16 MMA).
//   warps 4-7   softmax of tile 0, warps 8-11 softmax of tile 1: thread r owns row r
//               (TMEM lane r), S read whole (128 columns); exp2 with a log2(e)-folded
//               scale; P rounded to bf16 (d = 128: into the TMEM columns of S); O rescaled
//               only when the running max of a row that already holds probability mass
//               grows by more than 2^8 (exact: the final division uses the same stale
//               max).  Then the epilogue o = O / l.
//
// TMEM columns, d = 128: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512); P is
// packed bf16 in the first 64 columns of S_t.  d = 64: per tile t, S_t [256t, 256t+128),
// P_t [256t+128, 256t+192), O_t [256t+192, 256t+256).
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "moda_common.cuh"
#include "sm103_ptx.cuh"

namespace moda {
namespace {

using namespace sm103;

constexpr int BM = 128;                    // rows per query tile
constexpr int BN = 128;                    // keys per key tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kThreads = 384;
constexpr int kMaxG = 128;
constexpr int kSmemLimit = 232448;  // bytes of dynamic shared memory a CTA may use

// Shared memory: Q_0 | Q_1 | K/V ring (NSLOT tiles) | barriers, misc words.
template <int D>
struct FwdCfg {
  // As many slots as shared memory holds: in a unit's depth steps, which stream from HBM,
  // the bytes in flight per SM are what the ring has room for.
  static constexpr int NSLOT = D == 128 ? 5 : 12;
  static constexpr int TILE_BYTES = BM * D * 2;  // a Q, K or V tile: 128 rows x D bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_KV + NSLOT * TILE_BYTES;
  // kv_full[2 * NSLOT], kv_empty[NSLOT], q_full[2], q_empty[2], s_full[2], p_full[2],
  // pv_done[2], o_free[2], s_free[2], drain[2].  Each ring slot has two full barriers, used
  // by its even and odd loads: with one issuer per query tile an issuer can reach an item
  // whose slot still holds, not yet landed, an item only the other tile reads; the barrier
  // of its own item was last used two loads earlier, by a load every reader has consumed
  // (and so completed), so its parity wait cannot pass on an older load.
  static constexpr int NBAR = 3 * NSLOT + 16;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static_assert(SMEM <= kSmemLimit, "shared memory");
  // TMEM columns.  SPLIT (d = 64): S_t, P_t, O_t of tile t each in columns of their own,
  // [256t, +128), [256t + 128, +64), [256t + 192, +64), so S of the next key tile can be
  // computed while the softmax of this one still runs.  Otherwise (d = 128) there is room
  // for S and O only: P_t is packed into the first 64 columns of S_t, S_t at 128t, O_t at
  // 256 + 128t, and the next S waits until the PV that reads P was issued.
  static constexpr bool SPLIT = D == 64;
  static constexpr uint32_t tm_s(int t) { return SPLIT ? 256u * t : 128u * t; }
  static constexpr uint32_t tm_p(int t) { return SPLIT ? 256u * t + 128u : 128u * t; }
  static constexpr uint32_t tm_o(int t) { return SPLIT ? 256u * t + 192u : 256u + D * t; }
};

struct FwdTcParams {
  int B, H, Hkv, T, S, G, P;
  int Tk;       // keys per (b, kv head) in k/v (T unless a key chunk of another range is read)
  int delta;    // key j is visible to query position t iff j <= t + delta (0 <= delta)
  int S_read;   // slots read per position (the S - S_read others are never loaded)
  int n_pb;     // position blocks (of 2P positions) per (b, kv head)
  int n_units;  // B * Hkv * n_pb
  int n_cta;    // persistent CTAs
  int n_d;      // depth steps per query tile: ceil(S_read / 128) (0 without depth slots)
  int w;        // slots of a position per depth step: min(S_read, 128)
  int dpt;      // positions per depth chunk: floor(128 / w)
  int n_ch;     // depth chunks per depth step: ceil(P / dpt)
  int nd_keys;  // keys of a depth chunk's products: dpt * w rounded up to 16
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  int* status;
};

struct Unit {
  int b, g, bg, p0;
  int nt[2];     // sequence key tiles each query tile needs (0: tile beyond T)
  int ns[2];     // steps (depth + sequence key tiles) of each query tile (0: tile beyond T)
};

// Output-lane mask of TMEM rows [lo, hi) for a masked MMA: bit i of m[q] set leaves lane
// 32 q + i unwritten.
__device__ __forceinline__ void rows_mask(int lo, int hi, uint32_t (&m)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int a = min(max(lo - 32 * q, 0), 32), b = min(max(hi - 32 * q, 0), 32);
    const uint32_t below_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
    const uint32_t below_a = a >= 32 ? 0xffffffffu : ((1u << a) - 1u);
    m[q] = ~(below_b & ~below_a);
  }
}

// Units a CTA processes: the unit list in heaviest-first order, dealt round-robin with the
// direction reversed every round (snake), so every CTA gets a similar amount of work.
__device__ __forceinline__ int units_of_cta(const FwdTcParams& p, int c) {
  const int R = p.n_units / p.n_cta, rem = p.n_units % p.n_cta;
  const bool extra = (R & 1) ? (p.n_cta - 1 - c < rem) : (c < rem);
  return R + (extra ? 1 : 0);
}

__device__ __forceinline__ Unit unit_at(const FwdTcParams& p, int c, int k) {
  const int idx = k * p.n_cta + ((k & 1) ? p.n_cta - 1 - c : c);
  const int ngroups = p.B * p.Hkv;
  const int pb = p.n_pb - 1 - idx / ngroups;
  Unit u;
  u.bg = idx % ngroups;
  u.b = u.bg / p.Hkv;
  u.g = u.bg % p.Hkv;
  u.p0 = pb * 2 * p.P;
  const int end = min(u.p0 + 2 * p.P, p.T);
  const int nk = (p.Tk + BN - 1) / BN;  // key tiles of the key range
  u.nt[0] = min((min(u.p0 + p.P, p.T) - 1 + p.delta) / BN + 1, nk);
  u.nt[1] = (u.p0 + p.P < p.T) ? min((end - 1 + p.delta) / BN + 1, nk) : 0;
  u.ns[0] = p.n_d + u.nt[0];
  u.ns[1] = u.nt[1] > 0 ? p.n_d + u.nt[1] : 0;
  return u;
}

// K/V items of a unit, in the order the loader issues them (with per = n_ch * tw items of
// one kind per depth step, tw = 2 query tiles or 1 when tile 1 is empty):
//   depth step i:   the K items of the step's chunks, then their V items at + per.  With
//                   one MMA issuer per query tile (d = 64) the two tiles' chunks
//                   alternate (chunk c of tile t at 2 i per + c tw + t); the single issuer
//                   (d = 128) takes tile 0's chunks, then tile 1's (2 i per + t n_ch + c),
//                   so that tile 0's softmax starts while tile 1's products are issued;
//   sequence steps: K_j, V_j, each shared by both query tiles.
// With one issuer per tile (S of the next step issued before the P V of this one) the
// sequence's K_0 is hoisted between the K and the V items of the last depth step
// ("hoist"); the single issuer takes both tiles' depth P V before S of the next step, and
// K_0 stays in its place.
// Every consumer takes its items in load order, and an issuer's consecutive items are at
// most two apart within a unit (a unit's first item is waited for after its Q tile, which
// the loader issues after every item of the previous unit).  So when an issuer waits for
// item x, the loader has issued item x - NSLOT, which it does only after item x - 2 NSLOT
// was released: the earlier use of x's full barrier (even and odd loads of a slot have a
// barrier each) has completed, and the parity wait cannot pass on it.
struct Items {
  int base, tw, per, n_ch, n_d, hoist, nd;  // nd: items of the depth steps (with a hoisted K_0)
  bool tile_major;                          // the single issuer's order of a step's chunks
  __device__ __forceinline__ Items(const FwdTcParams& p, const Unit& u, int b, bool split)
      : base(b), tw(u.nt[1] > 0 ? 2 : 1), per(p.n_ch * tw), n_ch(p.n_ch), n_d(p.n_d),
        hoist(split && p.n_d > 0 ? 1 : 0), nd(p.n_d > 0 ? 2 * p.n_d * per + hoist : 0), tile_major(!split) {}
  __device__ __forceinline__ int chunk_off(int c, int t) const { return tile_major ? t * n_ch + c : c * tw + t; }
  __device__ __forceinline__ int dk(int i, int c, int t) const { return base + 2 * i * per + chunk_off(c, t); }
  __device__ __forceinline__ int dv(int i, int c, int t) const {
    return base + 2 * i * per + per + (i == n_d - 1 ? hoist : 0) + chunk_off(c, t);
  }
  __device__ __forceinline__ int sk(int j) const {
    return hoist ? (j == 0 ? base + 2 * (n_d - 1) * per + per : base + nd + 2 * j - 1) : base + nd + 2 * j;
  }
  __device__ __forceinline__ int sv(int j) const { return base + nd + 2 * j + 1 - hoist; }
  // first item of the next unit, after m sequence steps
  __device__ __forceinline__ int end(int m) const { return base + nd + 2 * m - hoist; }
  // what item r (from base) is: kind 0/1 depth K/V of step i, chunk c, tile t; 2/3
  // sequence K/V of step j
  __device__ __forceinline__ void decode(int r, int& kind, int& i, int& c, int& t, int& j) const {
    i = c = t = j = 0;
    if (r < nd) {
      i = min(r / (2 * per), n_d - 1);
      const int rem = r - 2 * i * per, lastd = i == n_d - 1 ? hoist : 0;
      if (lastd && rem == per) {
        kind = 2;  // the hoisted K_0
        return;
      }
      kind = rem < per ? 0 : 1;
      const int e = rem < per ? rem : rem - per - lastd;
      c = tile_major ? e % n_ch : e / tw;
      t = tile_major ? e / n_ch : e % tw;
    } else {
      const int q = r - nd + hoist;  // index in K_0 V_0 K_1 V_1 ...
      j = q >> 1;
      kind = 2 + (q & 1);
    }
  }
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    moda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKd,
                       const __grid_constant__ CUtensorMap tmVd, const FwdTcParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  // The 128-byte swizzle atoms need 1024-byte aligned tiles; the dynamic shared window
  // starts 1024-aligned on this architecture, and a launch where it does not is refused.
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int n_c = units_of_cta(p, cta);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;  // [2 * NSLOT]: slot s, load generation g -> kv_full[2s + (g & 1)]
  uint64_t* kv_empty = bars + 2 * C::NSLOT;
  uint64_t* q_full = bars + 3 * C::NSLOT;
  uint64_t* q_empty = q_full + 2;
  uint64_t* s_full = q_empty + 2;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_free = pv_done + 2;
  uint64_t* s_free = o_free + 2;
  uint64_t* drain = s_free + 2;
  uint8_t* misc = smem + C::OFF_BAR + C::NBAR * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(&kv_full[2 * i], 1);
      mbar_init(&kv_full[2 * i + 1], 1);
      mbar_init(&kv_empty[i], C::SPLIT ? 2 : 1);  // released by each MMA issuer
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_empty[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&pv_done[t], 1);
      mbar_init(&o_free[t], 128);
      mbar_init(&s_free[t], 4);  // one arrival per softmax warp (SPLIT)
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    if (p.S > 0) {
      prefetch_tmap(&tmKd);
      prefetch_tmap(&tmVd);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (p.n_d > 0 && p.dpt * p.w < p.nd_keys) {
    // rows of a depth chunk past its dpt * w keys are seen by no row, but enter the P V
    // product with P = 0: they must hold finite numbers, so the ring starts zeroed
    // (afterwards they hold loaded keys and values)
    for (int i = threadIdx.x; i < C::NSLOT * C::TILE_BYTES / 16; i += kThreads)
      st_shared_v4(sbase + C::OFF_KV + i * 16, make_uint4(0, 0, 0, 0));
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int it = 0, issued = 0, q_issued0 = 0, q_issued1 = 0;
      bool ok = true;
      // Q tiles and depth slabs are read once: evict first, so they do not displace the
      // sequence K/V that other query tiles read again
      const uint64_t pol_once = l2_policy_evict_first();
      for (int k = 0; ok && k < n_c; ++k) {
        const Unit u = unit_at(p, cta, k);
        for (int t = 0; ok && t < 2; ++t) {
          if (k > 0 && !mbar_wait(&q_empty[t], (k - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::OFF_Q + t * C::TILE_BYTES;
          mbar_arrive_expect_tx(&q_full[t], (D / 64) * p.G * p.P * 128);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d_hint(dst + h * (BM * 128), &tmQ, &q_full[t], h * 64, u.g * p.G, u.p0 + t * p.P, u.b,
                             pol_once);
          if (t == 0)
            q_issued0 = k + 1;
          else
            q_issued1 = k + 1;
        }
        const Items itl(p, u, 0, C::SPLIT);
        const int n_items = itl.end(max(u.nt[0], u.nt[1]));
        // d = 128: while this unit's sequence tiles load, one depth chunk of the next unit
        // per item is prefetched into L2 (the 5-slot ring holds few bytes in flight during
        // a depth step; at d = 64 the 12-slot ring does, and the prefetch only displaced
        // sequence K/V from L2)
        const bool pf_next = D == 128 && p.n_d > 0 && k + 1 < n_c;
        const Unit un = pf_next ? unit_at(p, cta, k + 1) : u;
        const Items itn(p, un, 0, C::SPLIT);
        int pf = 0;
        for (int r = 0; ok && r < n_items; ++r, ++it) {
          const int slot = it % C::NSLOT, use = it / C::NSLOT;
          if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::OFF_KV + slot * C::TILE_BYTES;
          uint64_t* full = &kv_full[2 * slot + (use & 1)];
          int kind, i, c, t, j;
          itl.decode(r, kind, i, c, t, j);
          if (kind < 2) {
            // depth chunk c of step i of tile t: dpt positions x w slots; rows past dpt * w
            // keep what the slot held (finite: zeroed at start, then loaded keys and values)
            // and are seen by no row
            const CUtensorMap* map = kind ? &tmVd : &tmKd;
            const int pos0 = u.bg * p.T + u.p0 + t * p.P + c * p.dpt;
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(D) * p.w * p.dpt * 2);
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d_hint(dst + h * (BN * 128), map, full, h * 64, i * BN, pos0, pol_once);
          } else {
            mbar_arrive_expect_tx(full, C::TILE_BYTES);
            const CUtensorMap* map = kind == 3 ? &tmV : &tmK;
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(dst + h * (BN * 128), map, full, h * 64, j * BN, u.bg);
          }
          if (pf_next && r >= itl.nd && pf < itn.nd) {
            // (at d = 128 the depth items are all of the next unit's first itn.nd items)
            int kn, in_, cn, tn, jn;
            itn.decode(pf++, kn, in_, cn, tn, jn);
            const CUtensorMap* mp = kn ? &tmVd : &tmKd;
            const int ps = un.bg * p.T + un.p0 + tn * p.P + cn * p.dpt;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) tma_prefetch_3d(mp, h * 64, in_ * BN, ps);
          }
          issued = it + 1;
        }
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        // let every copy still in flight land before the CTA exits
        volatile int never = 0;
        for (int i = max(0, issued - C::NSLOT); i < issued; ++i)
          mbar_wait(&kv_full[2 * (i % C::NSLOT) + ((i / C::NSLOT) & 1)], (i / C::NSLOT / 2) & 1, &never);
        if (q_issued0 > 0) mbar_wait(&q_full[0], (q_issued0 - 1) & 1, &never);
        if (q_issued1 > 0) mbar_wait(&q_full[1], (q_issued1 - 1) & 1, &never);
      }
    }
  } else if (!C::SPLIT && warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (d = 128)
    // One warp for both tiles (its elected lane issues): PV_0(i), S_0(i+1), PV_1(i), S_1(i+1)
    // in this order, since S of the next key tile overwrites P of this one.
    {
      constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false);
      constexpr uint32_t IDESC_O = idesc_bf16(BM, D, true);
      const uint32_t idesc_d = idesc_bf16(BM, p.nd_keys, false);  // a depth chunk's S
      const uint64_t q_desc0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t kv_desc_k = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);        // K-major (K tiles)
      const uint64_t kv_desc_v = sdesc_sw128(sbase + C::OFF_KV, BN * 128, 1024);  // MN-major (V tiles)
      int base = 0;                    // first item of the unit
      uint32_t pcnt0 = 0, pcnt1 = 0;  // p_full phases consumed per tile
      bool ok = true;
      auto wait_item = [&](int item) -> bool {
        const int g = item / C::NSLOT;  // load generation of the slot
        return warp_wait(&kv_full[2 * (item % C::NSLOT) + (g & 1)], (g >> 1) & 1, abort_flag);
      };
      auto release = [&](int item) { mma_commit_warp(&kv_empty[item % C::NSLOT]); };
      
      auto issue_s = [&](int t, int item) {
        const uint64_t q_desc = sdesc_add(q_desc0, t * C::TILE_BYTES);
        const uint64_t k_desc = sdesc_add(kv_desc_k, (item % C::NSLOT) * C::TILE_BYTES);
        const uint32_t d_tmem = tmem + C::tm_s(t);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss(d_tmem, sdesc_add(q_desc, (kk >> 2) * (BM * 128) + (kk & 3) * 32),
                        sdesc_add(k_desc, (kk >> 2) * (BN * 128) + (kk & 3) * 32), IDESC_S, kk > 0);
          mma_commit(&s_full[t]);
        }
        __syncwarp();
      };
      // pv_done is committed only after a tile's last PV of the unit (for its epilogue):
      // before that, S of the next key tile, issued after this PV, tells the softmax warps
      // that O is up to date (MMAs of one thread complete in order).
      auto issue_pv = [&](int t, int item, bool acc, bool last) {
        const uint64_t v_desc = sdesc_add(kv_desc_v, (item % C::NSLOT) * C::TILE_BYTES);
        const uint32_t p_tmem = tmem + C::tm_p(t);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_bf16_ts(tmem + C::tm_o(t), p_tmem + kk * 8, sdesc_add(v_desc, kk * 16 * 128), IDESC_O,
                        (acc || kk > 0) ? 1u : 0u);
          if (last) mma_commit(&pv_done[t]);
        }
        __syncwarp();
      };
      // The issuing warp is on the critical path between MMA groups: the depth and sequence
      // steps have a loop each.
      for (int k = 0; ok && k < n_c; ++k) {
        const Unit u = unit_at(p, cta, k);
        const int nA = u.ns[0], nB = u.ns[1];
        const bool two = nB > 0;
        ok = warp_wait(&q_full[0], k & 1, abort_flag) && warp_wait(&q_full[1], k & 1, abort_flag);
        if (!ok) break;
        if (!two) mma_commit_warp(&q_empty[1]);  // tile 1 unused in this unit
        const Items it(p, u, base, false);
        // S of depth step i of tile t: every chunk's product into S_t, masked to the
        // chunk's rows, then one commit
        auto depth_s = [&](int t, int i) -> bool {
          const uint64_t q_desc = sdesc_add(q_desc0, t * C::TILE_BYTES);
          for (int c = 0; c < p.n_ch; ++c) {
            const int item = it.dk(i, c, t);
            if (!wait_item(item)) return false;
            tc_fence_after();
            uint32_t mask[4];
            rows_mask(c * p.dpt * p.G, min((c + 1) * p.dpt, p.P) * p.G, mask);
            const uint64_t k_desc = sdesc_add(kv_desc_k, (item % C::NSLOT) * C::TILE_BYTES);
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_bf16_ss_mask(tmem + C::tm_s(t), sdesc_add(q_desc, (kk >> 2) * (BM * 128) + (kk & 3) * 32),
                                 sdesc_add(k_desc, (kk >> 2) * (BN * 128) + (kk & 3) * 32), idesc_d, kk > 0, mask);
            }
            __syncwarp();
            release(item);
          }
          mma_commit_warp(&s_full[t]);
          return true;
        };
        // O_t += P_t V of depth step i once P_t is written: each chunk's product masked to
        // the chunk's rows (step 0 starts each row's O)
        auto depth_pv = [&](int t, int i) -> bool {
          uint32_t& pc = t ? pcnt1 : pcnt0;
          if (!warp_wait(&p_full[t], pc & 1, abort_flag) ||
              (i == 0 && k > 0 && !warp_wait(&o_free[t], (k - 1) & 1, abort_flag)))
            return false;
          ++pc;
          tc_fence_after();
          for (int c = 0; c < p.n_ch; ++c) {
            const int item = it.dv(i, c, t);
            if (!wait_item(item)) return false;
            tc_fence_after();
            uint32_t mask[4];
            rows_mask(c * p.dpt * p.G, min((c + 1) * p.dpt, p.P) * p.G, mask);
            const uint64_t v_desc = sdesc_add(kv_desc_v, (item % C::NSLOT) * C::TILE_BYTES);
            if (elect_one()) {
              for (int kk = 0; kk < p.nd_keys / 16; ++kk)
                mma_bf16_ts_mask(tmem + C::tm_o(t), tmem + C::tm_p(t) + kk * 8, sdesc_add(v_desc, kk * 16 * 128),
                                 IDESC_O, (i > 0 || kk > 0) ? 1u : 0u, mask);
            }
            __syncwarp();
            release(item);
          }
          return true;
        };
        // S of step 0
        if (p.n_d > 0) {
          if (!depth_s(0, 0) || (two && !depth_s(1, 0))) {
            ok = false;
            break;
          }
        } else {
          if (!wait_item(it.sk(0))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(0, it.sk(0));
          if (nA == 1) mma_commit_warp(&q_empty[0]);
          if (two) {
            issue_s(1, it.sk(0));
            if (nB == 1) mma_commit_warp(&q_empty[1]);
          }
          release(it.sk(0));
        }
        // ---- depth steps: each query tile has K and V items of its own.  Tile 0's P V,
        // tile 1's, then S of step i+1 (the next depth step, or the first sequence step,
        // whose K both tiles read): the items are consumed in the order they are loaded.
        for (int i = 0; ok && i < p.n_d; ++i) {
          if (!depth_pv(0, i) || (two && !depth_pv(1, i))) {
            ok = false;
            break;
          }
          if (i + 1 < p.n_d) {
            if (!depth_s(0, i + 1) || (two && !depth_s(1, i + 1))) {
              ok = false;
              break;
            }
          } else {
            if (!wait_item(it.sk(0))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(0, it.sk(0));
            if (two) issue_s(1, it.sk(0));
            release(it.sk(0));
          }
          if (i + 2 == nA) mma_commit_warp(&q_empty[0]);
          if (two && i + 2 == nB) mma_commit_warp(&q_empty[1]);
        }
        // ---- sequence steps: K and V shared by both tiles; S of the first was issued above
        const int mA = nA - p.n_d, mB = two ? nB - p.n_d : 0, m = max(mA, mB);
        for (int j = 0; ok && j < m; ++j) {
          const int iv = it.sv(j), ik = it.sk(j + 1);
          const bool first = p.n_d == 0 && j == 0;  // first PV of the unit
          if (!wait_item(iv)) {
            ok = false;
            break;
          }
          if (j < mA) {
            if (!warp_wait(&p_full[0], pcnt0 & 1, abort_flag) ||
                (first && k > 0 && !warp_wait(&o_free[0], (k - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            ++pcnt0;
            tc_fence_after();
            issue_pv(0, iv, !first, j + 1 == mA);
          }
          const bool next = j + 1 < m;
          if (next && !wait_item(ik)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (j + 1 < mA) {
            issue_s(0, ik);
            if (j + 2 == mA) mma_commit_warp(&q_empty[0]);
          }
          if (j < mB) {
            if (!warp_wait(&p_full[1], pcnt1 & 1, abort_flag) ||
                (first && k > 0 && !warp_wait(&o_free[1], (k - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            ++pcnt1;
            tc_fence_after();
            issue_pv(1, iv, !first, j + 1 == mB);
          }
          release(iv);  // V_j: every PV reading it is issued
          if (j + 1 < mB) {
            issue_s(1, ik);
            if (j + 2 == mB) mma_commit_warp(&q_empty[1]);
          }
          if (next) release(ik);  // K_{j+1}: every S reading it is issued
        }
        base = it.end(m);
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        // wait for every MMA already issued before TMEM is released
        mma_commit_warp(&drain[0]);
        volatile int never = 0;
        mbar_wait(&drain[0], 0, &never);
      }
    }
  } else if (C::SPLIT && (warp == 1 || warp == 2)) {
    // ---------------------------------------------------------------- MMA issuers (d = 64)
    // One warp per query tile t (warps 1 and 2; the elected lane issues), so neither tile's
    // S/PV chain waits on the other's softmax.  Every K/V item is released twice: once by
    // each tile that uses it, twice by its only user otherwise.
    {
      const int t = warp - 1;
      constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false);
      constexpr uint32_t IDESC_O = idesc_bf16(BM, D, true);
      const uint32_t idesc_d = idesc_bf16(BM, p.nd_keys, false);  // a depth chunk's S
      const uint64_t q_desc = sdesc_sw128(sbase + C::OFF_Q + t * C::TILE_BYTES, 16, 1024);
      const uint64_t kv_desc_k = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);        // K-major (K tiles)
      const uint64_t kv_desc_v = sdesc_sw128(sbase + C::OFF_KV, BN * 128, 1024);  // MN-major (V tiles)
      const uint32_t s_tm = tmem + C::tm_s(t), p_tm = tmem + C::tm_p(t), o_tm = tmem + C::tm_o(t);
      int base = 0;                     // first item of the unit
      uint32_t scnt = 0, pcnt = 0;      // S issued, p_full phases consumed
      bool ok = true;
      auto wait_item = [&](int item) -> bool {
        const int g = item / C::NSLOT;  // load generation of the slot
        return warp_wait(&kv_full[2 * (item % C::NSLOT) + (g & 1)], (g >> 1) & 1, abort_flag);
      };
      auto release = [&](int item, bool shared) {
        if (elect_one()) {
          mma_commit(&kv_empty[item % C::NSLOT]);
          if (!shared) mma_commit(&kv_empty[item % C::NSLOT]);
        }
        __syncwarp();
      };
      auto issue_s = [&](int item) {
        const uint64_t k_desc = sdesc_add(kv_desc_k, (item % C::NSLOT) * C::TILE_BYTES);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ss(s_tm, sdesc_add(q_desc, (kk >> 2) * (BM * 128) + (kk & 3) * 32),
                        sdesc_add(k_desc, (kk >> 2) * (BN * 128) + (kk & 3) * 32), IDESC_S, kk > 0);
          mma_commit(&s_full[t]);
        }
        __syncwarp();
        ++scnt;
      };
      auto issue_pv = [&](int item, bool acc) {
        const uint64_t v_desc = sdesc_add(kv_desc_v, (item % C::NSLOT) * C::TILE_BYTES);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_bf16_ts(o_tm, p_tm + kk * 8, sdesc_add(v_desc, kk * 16 * 128), IDESC_O, (acc || kk > 0) ? 1u : 0u);
          mma_commit(&pv_done[t]);
        }
        __syncwarp();
      };
      for (int k = 0; ok && k < n_c; ++k) {
        const Unit u = unit_at(p, cta, k);
        const int n_t = t ? u.ns[1] : u.ns[0];
        const int nt_other = t ? u.nt[0] : u.nt[1];  // sequence tiles of the other query tile
        const Items it(p, u, base, true);
        // S of step i: a depth step's chunks (each masked to its rows, one commit), or the
        // sequence tile's K, read by the other tile too while it has that tile
        auto step_s = [&](int i) -> bool {
          if (i < p.n_d) {
            for (int c = 0; c < p.n_ch; ++c) {
              const int item = it.dk(i, c, t);
              if (!wait_item(item)) return false;
              tc_fence_after();
              uint32_t mask[4];
              rows_mask(c * p.dpt * p.G, min((c + 1) * p.dpt, p.P) * p.G, mask);
              const uint64_t k_desc = sdesc_add(kv_desc_k, (item % C::NSLOT) * C::TILE_BYTES);
              if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                  mma_bf16_ss_mask(s_tm, sdesc_add(q_desc, (kk >> 2) * (BM * 128) + (kk & 3) * 32),
                                   sdesc_add(k_desc, (kk >> 2) * (BN * 128) + (kk & 3) * 32), idesc_d, kk > 0, mask);
              }
              __syncwarp();
              release(item, false);
            }
            mma_commit_warp(&s_full[t]);
            ++scnt;
            return true;
          }
          const int ki = it.sk(i - p.n_d);
          if (!wait_item(ki)) return false;
          tc_fence_after();
          issue_s(ki);
          release(ki, i - p.n_d < nt_other);
          return true;
        };
        // PV of step i once P is written: per depth chunk, masked to its rows (step 0 starts
        // each row's O); then pv_done
        auto step_pv = [&](int i) -> bool {
          if (!warp_wait(&p_full[t], pcnt & 1, abort_flag) ||
              (i == 0 && k > 0 && !warp_wait(&o_free[t], (k - 1) & 1, abort_flag)))
            return false;
          ++pcnt;
          tc_fence_after();
          if (i < p.n_d) {
            for (int c = 0; c < p.n_ch; ++c) {
              const int item = it.dv(i, c, t);
              if (!wait_item(item)) return false;
              tc_fence_after();
              uint32_t mask[4];
              rows_mask(c * p.dpt * p.G, min((c + 1) * p.dpt, p.P) * p.G, mask);
              const uint64_t v_desc = sdesc_add(kv_desc_v, (item % C::NSLOT) * C::TILE_BYTES);
              if (elect_one()) {
                for (int kk = 0; kk < p.nd_keys / 16; ++kk)
                  mma_bf16_ts_mask(o_tm, p_tm + kk * 8, sdesc_add(v_desc, kk * 16 * 128), IDESC_O,
                                   (i > 0 || kk > 0) ? 1u : 0u, mask);
              }
              __syncwarp();
              release(item, false);
            }
            mma_commit_warp(&pv_done[t]);
            return true;
          }
          const int vi = it.sv(i - p.n_d);
          if (!wait_item(vi)) return false;
          tc_fence_after();
          issue_pv(vi, i > 0);
          release(vi, i - p.n_d < nt_other);
          return true;
        };
        ok = warp_wait(&q_full[t], k & 1, abort_flag);
        if (!ok) break;
        if (n_t == 0) {
          mma_commit_warp(&q_empty[t]);  // tile unused in this unit
        } else {
          // S of step 0
          if (scnt > 0 && !warp_wait(&s_free[t], (scnt - 1) & 1, abort_flag)) ok = false;
          if (ok) ok = step_s(0);
          if (ok && n_t == 1) mma_commit_warp(&q_empty[t]);
          for (int i = 0; ok && i < n_t; ++i) {
            // S of step i+1 as soon as the softmax has read S of step i (PV of step i goes
            // first when both are depth steps: step i+1's K items are loaded after step i's
            // V items)
            const bool pv_first = i + 1 < p.n_d;
            if (pv_first && !step_pv(i)) {
              ok = false;
              break;
            }
            if (i + 1 < n_t) {
              if (!warp_wait(&s_free[t], (scnt - 1) & 1, abort_flag) || !step_s(i + 1)) {
                ok = false;
                break;
              }
              if (i + 2 == n_t) mma_commit_warp(&q_empty[t]);
            }
            if (!pv_first && !step_pv(i)) {
              ok = false;
              break;
            }
          }
        }
        base = it.end(max(u.nt[0], u.nt[1]));
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        // wait for every MMA this thread issued before TMEM is released
        mma_commit_warp(&drain[t]);
        volatile int never = 0;
        mbar_wait(&drain[t], 0, &never);
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = (wq << 5) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tmem = tmem + lane_base + C::tm_s(t);
    const uint32_t p_tmem = tmem + lane_base + C::tm_p(t);
    const uint32_t o_tmem = tmem + lane_base + C::tm_o(t);
    const int pl = r / p.G, hl = r - pl * p.G;  // local position and head of row r
    const float sl2 = p.scale_log2;
    uint32_t scnt = 0, jcnt = 0;  // s_full phases consumed, PVs of this tile so far
    uint32_t ucnt = 0;            // units with keys for this tile so far (pv_done phases, d = 128)
    bool ok = true;
    for (int k = 0; ok && k < n_c; ++k) {
      const Unit u = unit_at(p, cta, k);
      const int n_t = t ? u.ns[1] : u.ns[0];
      const int pfirst = u.p0 + t * p.P;
      const int pos = pfirst + pl;
      const bool valid = n_t > 0 && pl < p.P && pos < p.T;
      float m_run = -INFINITY, l_run = 0.f;
      bool s_ready = false;  // d = 64: S of this step found complete during the previous one
      for (int j = 0; j < n_t; ++j) {
        if (!s_ready) {
          ok = warp_wait(&s_full[t], scnt & 1, abort_flag);
          if (!ok) break;
        }
        s_ready = false;
        ++scnt;
        tc_fence_after();
        const bool depth = j < p.n_d;
        int lo, hi;  // visible columns [lo, hi) of this row in this key tile
        if (depth) {
          // the row's own position's slots 128 j .. 128 j + w - 1 (those below S_read) in
          // its chunk: local position x of chunk x / dpt has keys [(x % dpt) w, + w)
          lo = valid ? (pl % p.dpt) * p.w : BN;
          hi = valid ? lo + min(p.w, p.S_read - j * BN) : BN;
        } else {
          // keys kb + c with c < hi are visible: c <= pos + delta - kb and kb + c < Tk
          const int kb = (j - p.n_d) * BN;
          lo = 0;
          hi = (kb + BN - 1 > pfirst + p.delta || kb + BN > p.Tk || !valid)
                   ? (valid ? min(pos + p.delta - kb + 1, p.Tk - kb) : 0)
                   : BN;
        }
        float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
        {
          // S read whole (d = 64: then handed back to the MMA issuer for the next key tile;
          // d = 128: P is written over it once every column is in registers)
          // the load also returns the row's maximum over the 128 columns, which is the row
          // max whenever no column of the row is masked
          uint32_t s[BN];
          float m_raw;
          tmem_ld128_max(s_tmem, s, m_raw);
          if constexpr (C::SPLIT) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[t]);
          }
          if (lo > 0 || hi < BN) {
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (c < lo || c >= hi) s[c] = __float_as_uint(-INFINITY);
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; c += 8) {
              mx0 = fmax3(mx0, __uint_as_float(s[c + 0]), __uint_as_float(s[c + 1]));
              mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
              mx2 = fmax3(mx2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
              mx3 = fmax3(mx3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
            }
            m_raw = fmax3(mx0, mx1, fmaxf(mx2, mx3));
          }
          const float m_tile = m_raw * sl2;
          // P_t is free once the previous PV of this tile completed (d = 128: S of this step,
          // issued after that PV, is complete, so it has)
          bool pv_waited = j == 0 || !C::SPLIT;
          const bool need = m_tile > m_run + kRescaleThreshold;  // includes the first keys of a row
          if (__any_sync(0xffffffffu, need)) {
            const float m_new = need ? fmaxf(m_run, m_tile) : m_run;
            // a row that holds no mass yet (m_run = -inf) needs no rescale of O or l
            const float corr = (m_run == -INFINITY || !need) ? 1.f : ex2(m_run - m_new);
            if (__any_sync(0xffffffffu, corr != 1.f)) {
              // the previous PV of this tile must have landed in O before it is rescaled
              if (!pv_waited) {
                ok = warp_wait(&pv_done[t], (jcnt - 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                pv_waited = true;
              }
#pragma unroll 1
              for (int c = 0; c < D / 16; ++c) {
                uint32_t o[16];
                tmem_ld16(o_tmem + c * 16, o);
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                tmem_st16(o_tmem + c * 16, o);
              }
            }
            l_run *= corr;
            m_run = m_new;
          }
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          // P of the whole tile into registers first: only its store has to wait for the
          // previous PV of this tile to have read P_t
          uint32_t pk[BN / 2];
          bool pv_ready = false, s_next = false;
#pragma unroll
          for (int c = 0; c < BN; c += 4) {
            if constexpr (C::SPLIT) {
              if (c == BN / 2) {
                // halfway through the exponentials, test (without waiting) whether the previous
                // PV has read P_t and whether S of the next key tile, issued when this one was
                // read, is complete: their latencies overlap the second half
                if (!pv_waited) pv_ready = mbar_test_wait(&pv_done[t], (jcnt - 1) & 1);
                if (j + 1 < n_t) s_next = mbar_test_wait(&s_full[t], scnt & 1);
              }
            }
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
          if (!pv_waited) {
            if (!__all_sync(0xffffffffu, pv_ready)) {
              ok = warp_wait(&pv_done[t], (jcnt - 1) & 1, abort_flag);
              if (!ok) break;
            }
            tc_fence_after();
          }
          tmem_st64(p_tmem, pk);
          if constexpr (C::SPLIT) s_ready = __all_sync(0xffffffffu, s_next);
        }
        if (!ok) break;
        l_run += (ls0 + ls1) + (ls2 + ls3);
        tc_fence_before();
        mbar_arrive(&p_full[t]);
        ++jcnt;
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      if (n_t > 0) {
        ok = warp_wait(&pv_done[t], (C::SPLIT ? jcnt - 1 : ucnt) & 1, abort_flag);
        if (!ok) break;
        ++ucnt;
        tc_fence_after();
        const float inv = (valid && l_run > 0.f) ? 1.f / l_run : 0.f;
        const int h = u.g * p.G + hl;
        __nv_bfloat16* orow =
            p.o + ((static_cast<int64_t>(u.b) * p.H + (valid ? h : 0)) * p.T + (valid ? pos : 0)) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t os[32];
          tmem_ld32(o_tmem + c * 32, os);
          uint32_t pk2[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            pk2[i >> 1] = pack_bf16(__uint_as_float(os[i]) * inv, __uint_as_float(os[i + 1]) * inv);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk2[4 * i], pk2[4 * i + 1], pk2[4 * i + 2], pk2[4 * i + 3]);
          }
        }
        if (valid && p.lse != nullptr)
          p.lse[(static_cast<int64_t>(u.b) * p.H + h) * p.T + pos] = (m_run + __log2f(l_run)) * kLn2;
      }
      tc_fence_before();
      mbar_arrive(&o_free[t]);
    }
    if (!ok) raise_abort(abort_flag, p.status);
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
}

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [groups = B*Hkv][T][D] bf16 as a 3-D tensor (D, T, groups); box 64 x 128 x 1.
bool make_kv_map(CUtensorMap* map, const void* base, int D, int T, int groups) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(groups)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BN), 1};
  return encode(map, base, 3, dims, strides, box);
}

// Depth slabs [B*Hkv*T positions][C slots][D] bf16 as a 3-D tensor (D, S_read, positions):
// slots from S_read on lie outside it and are never loaded (a box reaching past S_read, or
// past the last position, reads zeros there); box 64 x w x dpt (the w slots of the dpt
// positions of a depth chunk).
bool make_depth_map(CUtensorMap* map, const void* base, int D, int S_read, int C, int64_t npos, int w, int dpt) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S_read),
                              static_cast<cuuint64_t>(npos)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(C) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(w), static_cast<cuuint32_t>(dpt)};
  return encode(map, base, 3, dims, strides, box);
}

// Q [B][H][T][D] bf16 described as (D, H, T, B) -- heads before positions -- so that a
// box 64 x G x P x 1 lands position-major (row = position * G + head); positions past T
// read as zeros.
bool make_q_map(CUtensorMap* map, const void* base, int D, int T, int H, int B, int P, int G) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(T) * D * 2, static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H) * T * D * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(P), 1};
  return encode(map, base, 4, dims, strides, box);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

template <int D>
cudaError_t launch(const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D>;
  const Problem& pr = a.p;
  FwdTcParams p;
  p.B = pr.B;
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.T = pr.T;
  p.Tk = pr.Tk;
  p.delta = pr.delta;
  p.S = pr.S;
  p.S_read = pr.S_read;
  p.G = pr.G;
  p.P = BM / pr.G;
  p.n_pb = (pr.T + 2 * p.P - 1) / (2 * p.P);
  p.n_units = pr.B * pr.Hkv * p.n_pb;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  p.n_cta = std::min(p.n_units, sms);
  const bool depth = pr.S > 0 && pr.S_read > 0;
  p.w = depth ? std::min(pr.S_read, BN) : 1;
  p.dpt = BN / p.w;
  p.n_d = depth ? (pr.S_read + BN - 1) / BN : 0;
  p.n_ch = depth ? (p.P + p.dpt - 1) / p.dpt : 0;
  p.nd_keys = std::min(BN, (p.dpt * p.w + 15) / 16 * 16);
  p.scale_log2 = pr.scale_log2;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.status = a.status;
  CUtensorMap tq, tk, tv, tkd, tvd;
  if (!make_q_map(&tq, a.q, D, pr.T, pr.H, pr.B, p.P, pr.G) || !make_kv_map(&tk, a.k, D, pr.Tk, pr.B * pr.Hkv) ||
      !make_kv_map(&tv, a.v, D, pr.Tk, pr.B * pr.Hkv))
    return cudaErrorInvalidValue;
  if (depth) {
    const int64_t npos = static_cast<int64_t>(pr.B) * pr.Hkv * pr.T;
    if (!make_depth_map(&tkd, a.kd, D, pr.S_read, pr.S, npos, p.w, p.dpt) ||
        !make_depth_map(&tvd, a.vd, D, pr.S_read, pr.S, npos, p.w, p.dpt))
      return cudaErrorInvalidValue;
  } else {
    tkd = tk;  // never read
    tvd = tv;
  }
  static std::atomic<uint64_t> attr_set{0};
  cudaError_t e = ensure_dynamic_smem(moda_fwd_tc_kernel<D>, C::SMEM, attr_set);
  if (e != cudaSuccess) return e;
  moda_fwd_tc_kernel<D><<<p.n_cta, kThreads, C::SMEM, s>>>(tq, tk, tv, tkd, tvd, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

bool fwd_sm103_supported(const Problem& p) {
  // depth positions are addressed with 32-bit TMA coordinates
  const int64_t npos = static_cast<int64_t>(p.B) * p.Hkv * p.T;
  return (p.d == 64 || p.d == 128) && p.G >= 1 && p.G <= kMaxG && npos < (int64_t(1) << 31);
}

cudaError_t launch_fwd_sm103(const FwdArgs& a, cudaStream_t s) {
  return a.p.d == 64 ? launch<64>(a, s) : launch<128>(a, s);
}

}  // namespace moda
