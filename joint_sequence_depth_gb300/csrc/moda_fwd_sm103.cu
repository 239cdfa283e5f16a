// MoDA forward on the sm_103a tensor cores: a persistent kernel with two ping-pong
// query tiles per work unit, tcgen05 MMAs into TMEM fed by TMA, and the
// same-position depth slots folded in on the CUDA cores by warps of their own.
//
// Operation: "Mixture-of-Depths Attention", frame "One denominator allocates
// probability across both memories" (Sec. 2.2, Algorithm 1): one softmax over
// the causal sequence keys and the depth slots of the query's own position.
//
// Work unit.  256 expanded query rows of one (batch b, kv head g): two tiles of
// 128 rows, tile t holding the G query heads of g at the P = floor(128/G) positions
// p0 + t*P .. p0 + t*P + P - 1.  Inside a tile the rows are head-major,
// row r -> (head g*G + r/P, position p0 + t*P + r%P): the grouped row expansion of
// frame "Backup: grouped indexing preserves the correct token map" (T_q = G*T_kv),
// loaded by one 4-D TMA box (d, P positions, G heads).  Every K/V tile of kv head g
// is loaded once for the G heads and both tiles, and each position's [S, d] depth
// slab once for its G rows (the group-aware reuse of Sec. 3.2 / Fig. 4, without its
// packed layout).  Units are ordered heaviest first and dealt to the persistent CTAs
// in a snake order; each CTA alternates its heavy and light units so the depth
// stream (constant per unit) and the sequence loop (growing with the position) stay
// balanced.
//
// Warp roles (512 threads):
//   warp 0      TMA: the two Q tiles of each unit, then K_j, V_j tiles (128 keys) into
//               a ring of smem slots.
//   warp 1      TMEM allocator and MMA issuer (one thread).  Per key tile j:
//                 PV_0(j-1), S_0(j), PV_1(j-1), S_1(j)  with  S_t = Q_t K_j^T into TMEM
//                 S[t] and O_t += P_t V_j (P_t read from TMEM), so the tensor core works
//                 on one tile while the other tile's softmax runs.
//   warps 4-7   softmax of tile 0, warps 8-11 softmax of tile 1: thread r owns row r
//               (TMEM lane r); online softmax with running max m and denominator l
//               (frame "Shared online-softmax states preserve the joint operator"),
//               exp2 with a log2(e)-folded scale, P_j rounded to bf16 into the TMEM
//               columns of S_j, O rescaled only when the running max grows by more than
//               2^8 (exact: the final division uses the same stale max); then the
//               epilogue.
//   warps 12-15 depth: warp w takes every fourth position of each unit and streams its
//               depth K and V slab, in chunks of up to SC slots, by bulk copies into a
//               ring of its own; per chunk it computes the scores of the position's G rows
//               (lanes split slots x 16-byte chunks, fp32 accumulation of bf16 products,
//               cross-lane sums) and folds them into the running max m_d, sum l_d and
//               o_d = sum_i 2^(b_i - m_d) vd_i, which it leaves in a per-CTA scratch slot
//               that stays in L2.
// The epilogue merges the sequence state (m, l, O) with the depth state by the
// online-softmax update rule and divides once:
//   o = (2^(m-M) O + 2^(m_d-M) o_d) / (2^(m-M) l + 2^(m_d-M) l_d),  M = max(m, m_d),
// the single denominator of the joint operator.
//
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 [256+d,256+2d); P_j
// is packed bf16 in the first 64 columns of S_t.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "moda_common.cuh"
#include "sm103_ptx.cuh"

namespace moda {
namespace {

using namespace sm103;

constexpr int BM = 128;                    // rows per query tile
constexpr int BN = 128;                    // keys per K/V tile
constexpr int kUnitRows = 2 * BM;          // rows per work unit
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kThreads = 512;
constexpr int kDepthWarps = 4;
constexpr int kMaxNsw = 4;  // ring stages per depth warp
constexpr int kMaxS = 64;   // depth slots this kernel handles
constexpr int kMaxG = 8;    // query heads per kv head this kernel handles
constexpr int kSmemLimit = 232448;  // bytes of dynamic shared memory a CTA may use
constexpr int kMaxChunk = 32;  // depth slots per chunk
constexpr int kPbufBytes = 4 * kMaxG * kMaxChunk * 2;  // per depth warp: bf16 p[head][slot of the chunk]

// Shared memory: Q_0 | Q_1 | K/V ring (NSLOT tiles) | depth rings (4 warps x nsw stages,
// host-sized) | barriers, misc words, depth p-buffers.
template <int D>
struct FwdCfg {
  static constexpr int NSLOT = D == 128 ? 3 : 4;
  static constexpr int TILE_BYTES = BM * D * 2;  // a Q, K or V tile: 128 rows x D bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = 2 * TILE_BYTES;
  static constexpr int OFF_DEP = OFF_KV + NSLOT * TILE_BYTES;
  // kv_full[NSLOT], kv_empty[NSLOT], q_full[2], q_empty[2], s_full[2], p_full[2], pv_done[2],
  // o_free[2], dscr_full[2], dscr_empty[2][2], drain, dfull[kDepthWarps][kMaxNsw]
  static constexpr int NBAR = 2 * NSLOT + 18 + 1 + kDepthWarps * kMaxNsw;
  static constexpr int TAIL = NBAR * 8 + 32 + kPbufBytes;  // barriers, misc words, p-buffers (16-aligned)
  static constexpr uint32_t TM_O = 256;  // O_t at TM_O + t*D; S_t at t*BN
  static constexpr int off_bar(int ring) { return OFF_DEP + ring; }
  static constexpr int smem_bytes(int ring) { return off_bar(ring) + TAIL; }
  static constexpr int scratch_floats() { return kUnitRows * 2 + kUnitRows * D; }  // one slot
};

struct FwdTcParams {
  int B, H, Hkv, T, S, G, P;
  int n_pb;      // position blocks (of 2P positions) per (b, kv head)
  int n_units;   // B * Hkv * n_pb
  int n_cta;     // persistent CTAs
  int sc;       // depth slots per chunk
  int nck;      // chunks per position (ceil(S / sc))
  int nsw;      // ring stages per depth warp
  int dstage;   // bytes of one stage: Kd chunk then Vd chunk, each sc*D*2
  float scale_log2;
  const __nv_bfloat16* q;
  const __nv_bfloat16* kd;
  const __nv_bfloat16* vd;
  __nv_bfloat16* o;
  float* lse;
  float* scratch;  // per CTA: 2 slots of [256 x {m_d, l_d}] then o_d as [D/4][256 rows][4]
  int* status;
};

struct Unit {
  int b, g, bg, p0;
  int npos;    // valid positions (< T) of the unit
  int nt[2];   // key tiles each query tile needs (0: tile beyond T)
};

// Units a CTA processes: unit list in heaviest-first order, dealt round-robin with the
// direction reversed every round (snake), so every CTA gets a similar amount of work.
__device__ __forceinline__ int units_of_cta(const FwdTcParams& p, int c) {
  const int R = p.n_units / p.n_cta, rem = p.n_units % p.n_cta;
  const bool extra = (R & 1) ? (p.n_cta - 1 - c < rem) : (c < rem);
  return R + (extra ? 1 : 0);
}

// The k-th unit the CTA processes: its own list taken heavy, light, heavy, light, ...
__device__ __forceinline__ Unit unit_at(const FwdTcParams& p, int c, int k, int n_c) {
  const int i = (k & 1) ? n_c - 1 - (k >> 1) : (k >> 1);
  const int idx = i * p.n_cta + ((i & 1) ? p.n_cta - 1 - c : c);
  const int ngroups = p.B * p.Hkv;
  const int pb = p.n_pb - 1 - idx / ngroups;
  Unit u;
  u.bg = idx % ngroups;
  u.b = u.bg / p.Hkv;
  u.g = u.bg % p.Hkv;
  u.p0 = pb * 2 * p.P;
  const int end = min(u.p0 + 2 * p.P, p.T);
  u.npos = end - u.p0;
  u.nt[0] = (min(u.p0 + p.P, p.T) - 1) / BN + 1;
  u.nt[1] = (u.p0 + p.P < p.T) ? (end - 1) / BN + 1 : 0;
  return u;
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  record_status(status, kStatusTimeout);
}

// All lanes wait on the same barrier phase; the warp takes one decision.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Sum of a[0..N) across lane groups by transposition: at each step (partner lane^OFF)
// a lane keeps one half of its values and adds the partner's copy of that half.  After
// STEPS steps a[0 .. N>>STEPS) hold full sums; the lane's values start at index
// sum over steps of (lane & OFF_step ? N_step/2 : 0).
template <int N, int OFF, int STEPS>
__device__ __forceinline__ void xreduce(float* a, int lane) {
  if constexpr (STEPS > 0) {
    constexpr int H = N / 2;
    const bool up = (lane & OFF) != 0;
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const float send = up ? a[j] : a[j + H];
      const float keep = up ? a[j + H] : a[j];
      a[j] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
    }
    xreduce<H, OFF / 2, STEPS - 1>(a, lane);
  }
}

template <int NIC, int CH>
__device__ __forceinline__ float head_group_max(float x) {
#pragma unroll
  for (int off = 1; off < NIC; off <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
#pragma unroll
  for (int off = CH; off < 32; off <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}
template <int NIC, int CH>
__device__ __forceinline__ float head_group_sum(float x) {
#pragma unroll
  for (int off = 1; off < NIC; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
#pragma unroll
  for (int off = CH; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Reduction over the lanes of one query head (X lanes, lane bits below log2 X) of SCP
// per-slot partial sums.  Transposing steps (partner lane^OFF keeps one half of the
// values and adds the partner's copy of it) while more than one value is left, then
// butterfly steps: afterwards a lane holds SCP / min(SCP, X) full sums, those of slots
// base(lane) + j, where each transposing step with (lane & OFF) set adds half of the
// values left before it.
template <int N, int OFF>
__device__ __forceinline__ void head_reduce(float* a, int lane) {
  if constexpr (OFF > 0) {
    if constexpr (N >= 2) {
      constexpr int H = N / 2;
      const bool up = (lane & OFF) != 0;
#pragma unroll
      for (int j = 0; j < H; ++j) {
        const float send = up ? a[j] : a[j + H];
        const float keep = up ? a[j + H] : a[j];
        a[j] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
      }
      head_reduce<H, OFF / 2>(a, lane);
    } else {
      a[0] += __shfl_xor_sync(0xffffffffu, a[0], OFF);
      head_reduce<1, OFF / 2>(a, lane);
    }
  }
}

// Depth part of one position (one warp), streamed over chunks of up to SCP slots with the
// online-softmax update between chunks (Algorithm 1 applied to the depth slots).
// Lane = (head hl = lane / X, part x = lane % X): the lane owns E = D/X consecutive
// columns of head hl, so per slot it forms a partial dot over its columns (all slots
// independent), and in the V pass it owns o[hl][its E columns] outright.
//   K pass: sc[s] = q[hl][cols] . kd[s][cols] for the chunk's slots; head_reduce over the
//     X lanes of the head leaves full scores spread over the lanes.
//   softmax statistics: running max m and sum l of head hl (log2 units); p = 2^(b - m)
//     rounded to bf16 into this warp's p-buffer [head][slot].
//   V pass: o[e] = o[e] * corr + sum_s p[hl][s] * vd[s][cols], bf16 x bf16 -> fp32.
template <int D, int X>
struct DepthState {
  static constexpr int E = D / X;  // columns per lane
  static constexpr int NQ = E / 2; // bf16 pairs per lane
  static constexpr int GS = E >= 32 ? 1 : 4;  // slots interleaved per step
  uint32_t q[NQ];
  uint32_t qn[NQ];  // q of the next position, loaded one position ahead
  float m, l;
  float o[E];

  // E bf16 (E/2 words) of a row part in shared memory (plain loads the compiler can schedule).
  __device__ __forceinline__ static void lds_part(const uint8_t* ptr, uint32_t (&w)[NQ]) {
    if constexpr (E >= 8) {
#pragma unroll
      for (int i = 0; i < E / 8; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(ptr)[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
    } else if constexpr (E == 4) {
      const uint2 v = *reinterpret_cast<const uint2*>(ptr);
      w[0] = v.x;
      w[1] = v.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t*>(ptr);
    }
  }

  __device__ __forceinline__ void load_q(const FwdTcParams& p, const Unit& u, int pos, bool active, int hl, int x) {
    if (active) {
      const int h = u.g * p.G + hl;
      const __nv_bfloat16* src = p.q + ((static_cast<int64_t>(u.b) * p.H + h) * p.T + pos) * D + x * E;
      if constexpr (E >= 8) {
#pragma unroll
        for (int i = 0; i < E / 8; ++i) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
          qn[4 * i] = v.x;
          qn[4 * i + 1] = v.y;
          qn[4 * i + 2] = v.z;
          qn[4 * i + 3] = v.w;
        }
      } else if constexpr (E == 4) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
        qn[0] = v.x;
        qn[1] = v.y;
      } else {
        qn[0] = __ldg(reinterpret_cast<const uint32_t*>(src));
      }
    } else {
#pragma unroll
      for (int i = 0; i < NQ; ++i) qn[i] = 0u;
    }
  }

  // Starts a position with the prefetched q.
  __device__ __forceinline__ void begin() {
#pragma unroll
    for (int i = 0; i < NQ; ++i) q[i] = qn[i];
    m = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) o[i] = 0.f;
  }

  // Slots [0, nsl) of the chunk at kbase / vbase (slot rows of D bf16), nsl <= SCP.
  template <int SCP>
  __device__ __forceinline__ void chunk(const FwdTcParams& p, int nsl, const uint8_t* kbase, const uint8_t* vbase,
                                        uint8_t* pbuf, int hl, int x, int lane) {
    constexpr int TS = (SCP < X) ? SCP : X;  // lanes the transposing steps spread slots over
    constexpr int NF = SCP / TS;             // full scores a lane holds afterwards
    const int coff = x * (E * 2);
    float sc[SCP];
    // K pass: GS slots at a time, their loads first, then interleaved dot chains
#pragma unroll
    for (int s0 = 0; s0 < SCP; s0 += GS) {
      uint32_t w[GS][NQ];
#pragma unroll
      for (int g = 0; g < GS; ++g) {
        if (s0 + g < nsl) {
          lds_part(kbase + (s0 + g) * (D * 2) + coff, w[g]);
        } else {
#pragma unroll
          for (int i = 0; i < NQ; ++i) w[g][i] = 0u;
        }
      }
      float a0[GS], a1[GS];
#pragma unroll
      for (int g = 0; g < GS; ++g) a0[g] = a1[g] = 0.f;
#pragma unroll
      for (int i = 0; i < NQ; i += 2) {
#pragma unroll
        for (int g = 0; g < GS; ++g) {
          a0[g] = dot2_bf16(q[i], w[g][i], a0[g]);
          if (i + 1 < NQ) a1[g] = dot2_bf16(q[i + 1], w[g][i + 1], a1[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < GS; ++g) sc[s0 + g] = a0[g] + a1[g];
    }
    head_reduce<SCP, X / 2>(sc, lane);
    // slot of value j: base + j, base from the transposing steps (high lane bits of x first)
    int base = 0;
    {
      int n = SCP;
#pragma unroll
      for (int off = X / 2; off >= 1; off >>= 1) {
        if (n >= 2) {
          if (x & off) base += n / 2;
          n /= 2;
        }
      }
    }
    const float sl2 = p.scale_log2;
    float cmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < NF; ++j) {
      sc[j] = (base + j < nsl) ? sc[j] * sl2 : -INFINITY;
      cmax = fmaxf(cmax, sc[j]);
    }
    // max and sum over the lanes holding distinct slots of this head (the transposing bits)
#pragma unroll
    for (int off = X / 2, n = SCP; off >= 1 && n >= 2; off >>= 1, n >>= 1)
      cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, off));
    const float m_new = fmaxf(m, cmax);
    const float corr = (m == -INFINITY) ? 0.f : ex2(m - m_new);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    float ls = 0.f;
    __nv_bfloat16* prow = reinterpret_cast<__nv_bfloat16*>(pbuf) + hl * kMaxChunk;
#pragma unroll
    for (int j = 0; j < NF; ++j) {
      const float e = ex2(sc[j] - m_use);
      ls += e;
      if (base + j < nsl) prow[base + j] = __float2bfloat16_rn(e);
    }
#pragma unroll
    for (int off = X / 2, n = SCP; off >= 1 && n >= 2; off >>= 1, n >>= 1)
      ls += __shfl_xor_sync(0xffffffffu, ls, off);
    l = l * corr + ls;
    m = m_new;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= corr;
    __syncwarp();
    // V pass: 8 p values of this head at a time, GS slots' loads ahead of their FMAs
#pragma unroll
    for (int s8 = 0; s8 < SCP; s8 += 8) {
      if (s8 < nsl) {
        const uint4 pv = *reinterpret_cast<const uint4*>(prow + s8);
        const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int s0 = s8; s0 < s8 + 8; s0 += GS) {
          uint32_t w[GS][NQ];
#pragma unroll
          for (int g = 0; g < GS; ++g) {
            if (s0 + g < nsl) {
              lds_part(vbase + (s0 + g) * (D * 2) + coff, w[g]);
            } else {
#pragma unroll
              for (int i = 0; i < NQ; ++i) w[g][i] = 0u;  // p of a missing slot may be stale: v = 0
            }
          }
#pragma unroll
          for (int g = 0; g < GS; ++g) {
            const int s = s0 + g - s8;
            const uint32_t pp = (s0 + g < nsl) ? pw[s >> 1] : 0u;
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
              if (s & 1)
                axpy2_bf16_hi(pp, w[g][i], o[2 * i], o[2 * i + 1]);
              else
                axpy2_bf16(pp, w[g][i], o[2 * i], o[2 * i + 1]);
            }
          }
        }
      }
    }
    __syncwarp();  // the p-buffer is rewritten by the next chunk
  }

  // (m, l) and o of row (head hl, position kpos) into the scratch slot.
  __device__ __forceinline__ void finish(const FwdTcParams& p, int kpos, bool active, int hl, int x, float* scr) {
    if (!active) return;
    const int tile = kpos / p.P, pl = kpos - tile * p.P;
    const int row = tile * BM + hl * p.P + pl;
    float* od = scr + kUnitRows * 2;
    if constexpr (E >= 4) {
#pragma unroll
      for (int i = 0; i < E; i += 4) {
        const int col = x * E + i;
        *reinterpret_cast<float4*>(od + ((col >> 2) * kUnitRows + row) * 4) =
            make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
      }
    } else {
      const int col = x * E;
      *reinterpret_cast<float2*>(od + ((col >> 2) * kUnitRows + row) * 4 + (col & 3)) = make_float2(o[0], o[1]);
    }
    if (x == 0) *reinterpret_cast<float2*>(scr + 2 * row) = make_float2(m, l);
  }
};

// Items of depth warp w: positions kpos = w, w+4, ... of each unit (in the CTA's unit
// order), each in chunks ck = 0 .. nck-1 of SC slots.
struct DepthIter {
  int k, kpos, ck;
  Unit u;
  // moves to the first unit from k on that has a position for warp w (kpos = w there)
  __device__ __forceinline__ void seek(const FwdTcParams& p, int cta, int n_c, int w) {
    for (; k < n_c; ++k) {
      u = unit_at(p, cta, k, n_c);
      if (w < u.npos) break;
    }
    kpos = w;
  }
  __device__ __forceinline__ void start(const FwdTcParams& p, int cta, int n_c, int w) {
    k = 0;
    ck = 0;
    seek(p, cta, n_c, w);
  }
  // next position (first chunk)
  __device__ __forceinline__ void next_pos(const FwdTcParams& p, int cta, int n_c, int w) {
    ck = 0;
    kpos += 4;
    if (kpos >= u.npos) {
      ++k;
      seek(p, cta, n_c, w);
    }
  }
  __device__ __forceinline__ void next(const FwdTcParams& p, int cta, int n_c, int w) {
    if (++ck < p.nck) return;
    next_pos(p, cta, n_c, w);
  }
};

// Depth warp w: its own ring of nsw stages (Kd chunk | Vd chunk), filled by its own lane 0
// up to nsw items ahead; the chunks of a position are folded in order, and each unit's
// results go to scratch slot k & 1 once the epilogue of unit k-2 has read it.
template <int D, int X, int SCP>
__device__ __forceinline__ void depth_warp(const FwdTcParams& p, int cta, int n_c, int w, int lane,
                                           const uint8_t* ring_ptr, uint64_t* dfull, uint64_t* dscr_full,
                                           uint64_t* dscr_empty, uint8_t* pbuf, float* scr_cta, int scr_floats,
                                           volatile int* abort_flag) {
  const uint32_t ring = smem_u32(ring_ptr);
  const int half = p.dstage / 2;
  const uint64_t pol = l2_policy_evict_first();
  DepthIter is;  // issue pointer
  is.start(p, cta, n_c, w);
  int issued = 0;
  auto issue = [&](int idx) {
    if (lane == 0) {
      const int s0 = is.ck * p.sc, nsl = min(p.sc, p.S - s0);
      const uint32_t bytes = static_cast<uint32_t>(nsl * D * 2);
      const int64_t src = ((static_cast<int64_t>(is.u.bg) * p.T + is.u.p0 + is.kpos) * p.S + s0) * D;
      const int slot = idx % p.nsw;
      const uint32_t dst = ring + slot * p.dstage;
      mbar_arrive_expect_tx(&dfull[slot], 2 * bytes);
      bulk_load_hint(dst, p.kd + src, bytes, &dfull[slot], pol);
      bulk_load_hint(dst + half, p.vd + src, bytes, &dfull[slot], pol);
    }
    is.next(p, cta, n_c, w);
  };
  while (issued < p.nsw && is.k < n_c) issue(issued++);

  DepthState<D, X> st;
  const int hl = lane / X, x = lane % X;
  const bool active = hl < p.G;
  DepthIter qi;  // position whose q is prefetched
  qi.start(p, cta, n_c, w);
  if (qi.k < n_c) st.load_q(p, qi.u, qi.u.p0 + qi.kpos, active, hl, x);
  int consumed = 0;
  bool ok = true;
  for (int k = 0; ok && k < n_c; ++k) {
    const Unit u = unit_at(p, cta, k, n_c);
    const int slot = k & 1;
    float* scr = scr_cta + slot * scr_floats;
    if (k >= 2) {
      const uint32_t par = ((k >> 1) - 1) & 1;
      ok = warp_wait(&dscr_empty[2 * slot], par, abort_flag) && warp_wait(&dscr_empty[2 * slot + 1], par, abort_flag);
      if (!ok) break;
    }
    for (int kpos = w; ok && kpos < u.npos; kpos += 4) {
      st.begin();
      qi.next_pos(p, cta, n_c, w);
      if (qi.k < n_c) st.load_q(p, qi.u, qi.u.p0 + qi.kpos, active, hl, x);
      for (int ck = 0; ck < p.nck; ++ck) {
        const int rs = consumed % p.nsw;
        ok = warp_wait(&dfull[rs], (consumed / p.nsw) & 1, abort_flag);
        if (!ok) break;
        const uint8_t* kb = ring_ptr + rs * p.dstage;
        st.template chunk<SCP>(p, min(p.sc, p.S - ck * p.sc), kb, kb + half, pbuf, hl, x, lane);
        ++consumed;
        // the slot is free again: refill it with this warp's next item
        fence_proxy_async_smem();
        __syncwarp();
        if (is.k < n_c) issue(issued++);
      }
      if (ok) st.finish(p, kpos, active, hl, x, scr);
    }
    if (!ok) break;
    __threadfence_block();
    __syncwarp();
    if (lane == 0) mbar_arrive(&dscr_full[slot]);
  }
  if (!ok) {
    raise_abort(abort_flag, p.status);
    // let this warp's copies still in flight land before the CTA exits
    volatile int never = 0;
    for (int i = consumed; i < issued; ++i) mbar_wait(&dfull[i % p.nsw], (i / p.nsw) & 1, &never);
  }
}

template <int D, int X>
__device__ __forceinline__ void depth_warp_x(const FwdTcParams& p, int cta, int n_c, int w, int lane,
                                             const uint8_t* ring, uint64_t* dfull, uint64_t* dscr_full,
                                             uint64_t* dscr_empty, uint8_t* pbuf, float* scr_cta, int scr_floats,
                                             volatile int* abort_flag) {
  if (p.sc <= 16)
    depth_warp<D, X, 16>(p, cta, n_c, w, lane, ring, dfull, dscr_full, dscr_empty, pbuf, scr_cta, scr_floats,
                         abort_flag);
  else
    depth_warp<D, X, 32>(p, cta, n_c, w, lane, ring, dfull, dscr_full, dscr_empty, pbuf, scr_cta, scr_floats,
                         abort_flag);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    moda_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdTcParams p) {
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
  const int ring = kDepthWarps * p.nsw * p.dstage;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::off_bar(ring));
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::NSLOT;
  uint64_t* q_full = bars + 2 * C::NSLOT;
  uint64_t* q_empty = q_full + 2;
  uint64_t* s_full = q_empty + 2;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_free = pv_done + 2;
  uint64_t* dscr_full = o_free + 2;
  uint64_t* dscr_empty = dscr_full + 2;  // [slot][tile]
  uint64_t* drain = dscr_empty + 4;
  uint64_t* dfull = drain + 1;
  uint8_t* misc = smem + C::off_bar(ring) + C::NBAR * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  uint8_t* pbuf_base = smem + ((C::off_bar(ring) + C::NBAR * 8 + 16 + 15) & ~15);
  float* scr_cta = p.scratch + static_cast<int64_t>(cta) * 2 * C::scratch_floats();

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_empty[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&pv_done[t], 1);
      mbar_init(&o_free[t], 128);
      mbar_init(&dscr_full[t], 4);
      mbar_init(&dscr_empty[2 * t], 4);
      mbar_init(&dscr_empty[2 * t + 1], 4);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kDepthWarps * kMaxNsw; ++i) mbar_init(&dfull[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (Q, K, V)
    if (lane == 0) {
      int it = 0, issued = 0, q_issued[2] = {0, 0};
      bool ok = true;
      for (int k = 0; ok && k < n_c; ++k) {
        const Unit u = unit_at(p, cta, k, n_c);
        for (int t = 0; ok && t < 2; ++t) {
          if (k > 0 && !mbar_wait(&q_empty[t], (k - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::OFF_Q + t * C::TILE_BYTES;
          mbar_arrive_expect_tx(&q_full[t], (D / 64) * p.P * p.G * 128);
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_load_4d(dst + h * (BM * 128), &tmQ, &q_full[t], h * 64, u.p0 + t * p.P, u.g * p.G, u.b);
          q_issued[t] = k + 1;
        }
        const int n = max(u.nt[0], u.nt[1]);
        for (int j = 0; ok && j < n; ++j) {
          for (int kind = 0; kind < 2; ++kind, ++it) {
            const int slot = it % C::NSLOT, use = it / C::NSLOT;
            if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            const CUtensorMap* map = kind ? &tmV : &tmK;
            uint8_t* dst = smem + C::OFF_KV + slot * C::TILE_BYTES;
            mbar_arrive_expect_tx(&kv_full[slot], C::TILE_BYTES);
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(dst + h * (BN * 128), map, &kv_full[slot], h * 64, j * BN, u.bg);
            issued = it + 1;
          }
        }
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        // let every copy still in flight land before the CTA exits
        volatile int never = 0;
        for (int i = max(0, issued - C::NSLOT); i < issued; ++i)
          mbar_wait(&kv_full[i % C::NSLOT], (i / C::NSLOT) & 1, &never);
        for (int t = 0; t < 2; ++t)
          if (q_issued[t] > 0) mbar_wait(&q_full[t], (q_issued[t] - 1) & 1, &never);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false);
      constexpr uint32_t IDESC_O = idesc_bf16(BM, D, true);
      const uint64_t q_desc0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
      const uint64_t kv_desc_k = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);        // K-major (K tiles)
      const uint64_t kv_desc_v = sdesc_sw128(sbase + C::OFF_KV, BN * 128, 1024);  // MN-major (V tiles)
      int it = 0;                // K/V item counter (K_j = 2j, V_j = 2j+1 within a unit)
      uint32_t pcnt[2] = {0, 0};  // p_full phases consumed per tile
      bool ok = true;
      auto wait_item = [&](int item) -> bool {
        return mbar_wait(&kv_full[item % C::NSLOT], (item / C::NSLOT) & 1, abort_flag);
      };
      auto issue_s = [&](int t, int item) {
        const uint64_t q_desc = sdesc_add(q_desc0, t * C::TILE_BYTES);
        const uint64_t k_desc = sdesc_add(kv_desc_k, (item % C::NSLOT) * C::TILE_BYTES);
        const uint32_t d_tmem = tmem + t * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(d_tmem, sdesc_add(q_desc, (kk >> 2) * (BM * 128) + (kk & 3) * 32),
                      sdesc_add(k_desc, (kk >> 2) * (BN * 128) + (kk & 3) * 32), IDESC_S, kk > 0);
        mma_commit(&s_full[t]);
      };
      auto issue_pv = [&](int t, int item, bool acc) {
        const uint64_t v_desc = sdesc_add(kv_desc_v, (item % C::NSLOT) * C::TILE_BYTES);
        const uint32_t p_tmem = tmem + t * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts(tmem + C::TM_O + t * D, p_tmem + kk * 8, sdesc_add(v_desc, kk * 16 * 128), IDESC_O,
                      (acc || kk > 0) ? 1u : 0u);
        mma_commit(&pv_done[t]);
      };
      for (int k = 0; ok && k < n_c; ++k) {
        const Unit u = unit_at(p, cta, k, n_c);
        const int nA = u.nt[0], nB = u.nt[1], n = max(nA, nB);
        const int base = it;
        ok = mbar_wait(&q_full[0], k & 1, abort_flag) && mbar_wait(&q_full[1], k & 1, abort_flag);
        if (!ok) break;
        if (nB == 0) mma_commit(&q_empty[1]);  // tile 1 unused in this unit
        // S_0(0), S_1(0)
        if (!wait_item(base)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(0, base);
        if (nA == 1) mma_commit(&q_empty[0]);
        if (nB > 0) {
          issue_s(1, base);
          if (nB == 1) mma_commit(&q_empty[1]);
        }
        mma_commit(&kv_empty[base % C::NSLOT]);
        for (int j = 0; ok && j < n; ++j) {
          const int iv = base + 2 * j + 1, ik = base + 2 * j + 2;
          // PV_0(j), then S_0(j+1) (P_0(j) lives in S_0's columns: in-order execution
          // makes the overwrite safe once PV_0(j) is issued)
          if (!wait_item(iv)) {
            ok = false;
            break;
          }
          if (j < nA) {
            if (!mbar_wait(&p_full[0], pcnt[0] & 1, abort_flag) ||
                (j == 0 && k > 0 && !mbar_wait(&o_free[0], (k - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            ++pcnt[0];
            tc_fence_after();
            issue_pv(0, iv, j > 0);
          }
          const bool next = j + 1 < n;
          if (next && !wait_item(ik)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (j + 1 < nA) {
            issue_s(0, ik);
            if (j + 2 == nA) mma_commit(&q_empty[0]);
          }
          // PV_1(j), then S_1(j+1)
          if (j < nB) {
            if (!mbar_wait(&p_full[1], pcnt[1] & 1, abort_flag) ||
                (j == 0 && k > 0 && !mbar_wait(&o_free[1], (k - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            ++pcnt[1];
            tc_fence_after();
            issue_pv(1, iv, j > 0);
          }
          mma_commit(&kv_empty[iv % C::NSLOT]);  // V_j: every PV reading it is issued
          if (j + 1 < nB) {
            issue_s(1, ik);
            if (j + 2 == nB) mma_commit(&q_empty[1]);
          }
          if (next) mma_commit(&kv_empty[ik % C::NSLOT]);  // K_{j+1}: every S reading it is issued
        }
        it = base + 2 * n;
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        // wait for every MMA already issued before TMEM is released
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
      }
    }
  }
  } else if (warp < 12) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int t = (warp - 4) >> 2;
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tmem + lane_base + t * BN;
    const uint32_t o_tmem = tmem + lane_base + C::TM_O + t * D;
    const int hl = r / p.P, pl = r - hl * p.P;
    const float sl2 = p.scale_log2;
    uint32_t scnt = 0, jcnt = 0;  // s_full phases consumed, PVs of this tile so far
    bool ok = true;
    for (int k = 0; ok && k < n_c; ++k) {
      const Unit u = unit_at(p, cta, k, n_c);
      const int n_t = u.nt[t];
      const int pfirst = u.p0 + t * p.P;
      const int pos = pfirst + pl;
      const bool valid = n_t > 0 && hl < p.G && pos < p.T;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_t; ++j) {
        ok = warp_wait(&s_full[t], scnt & 1, abort_flag);
        if (!ok) break;
        ++scnt;
        tc_fence_after();
        const int kb = j * BN;
        const bool masked = kb + BN - 1 > pfirst || !valid;  // diagonal tile or dead row
        float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
        // Two halves of 64 keys.  P of the first half is written (over S columns already
        // read) before the second half is loaded; if the second half raises the running max
        // past the threshold, the first half's P is rescaled in place with O and l.
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t s[64];
          tmem_ld64(s_tmem + half * 64, s);
          if (masked) {
            const int lim = valid ? pos - kb - half * 64 : -1;
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c > lim) s[c] = __float_as_uint(-INFINITY);
          }
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            mx0 = fmax3(mx0, __uint_as_float(s[c + 0]), __uint_as_float(s[c + 1]));
            mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
            mx2 = fmax3(mx2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
            mx3 = fmax3(mx3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
          }
          const float m_h = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
          if (j == 0 && half == 0) {
            m_run = m_h;
          } else if (__any_sync(0xffffffffu, m_h > m_run + kRescaleThreshold)) {
            const float m_new = fmaxf(m_run, m_h);
            const float corr = (m_run == -INFINITY) ? 1.f : ex2(m_run - m_new);
            if (j > 0) {
              // the previous PV of this tile must have landed in O before it is rescaled
              ok = warp_wait(&pv_done[t], (jcnt - 1) & 1, abort_flag);
              if (!ok) break;
              tc_fence_after();
#pragma unroll 1
              for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(o_tmem + c * 32, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
                tmem_st32(o_tmem + c * 32, o);
              }
            }
            if (half == 1) {
              // P of the first half, already in TMEM, was taken against the old max
              uint32_t pw[32];
              tmem_ld32(s_tmem, pw);
#pragma unroll
              for (int i = 0; i < 32; ++i) pw[i] = pack_bf16(bf16_lo(pw[i]) * corr, bf16_hi(pw[i]) * corr);
              tmem_st32(s_tmem, pw);
            }
            l_run *= corr;
            ls0 *= corr;
            ls1 *= corr;
            ls2 *= corr;
            ls3 *= corr;
            m_run = m_new;
          }
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
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
          tmem_st32(s_tmem + half * 32, pk);
        }
        if (!ok) break;
        l_run += (ls0 + ls1) + (ls2 + ls3);
        tc_fence_before();
        mbar_arrive(&p_full[t]);
        ++jcnt;
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      const int slot = k & 1;
      float* scr = scr_cta + slot * C::scratch_floats();
      if (n_t > 0) {
        ok = warp_wait(&pv_done[t], (jcnt - 1) & 1, abort_flag);
        if (ok && p.S > 0) ok = warp_wait(&dscr_full[slot], (k >> 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const int row = t * BM + r;
        float md = -INFINITY, ldp = 0.f;
        if (p.S > 0 && valid) {
          const float2 st = __ldcg(reinterpret_cast<const float2*>(scr) + row);
          md = st.x;
          ldp = st.y;
        }
        const float m = fmaxf(m_run, md);
        const float a_s = (l_run > 0.f) ? ex2(m_run - m) : 0.f;
        const float a_d = (ldp > 0.f) ? ex2(md - m) : 0.f;
        const float L = l_run * a_s + ldp * a_d;
        const float inv = valid ? 1.f / L : 0.f;
        const float ws = a_s * inv, wd = a_d * inv;
        const int h = u.g * p.G + hl;
        __nv_bfloat16* orow =
            p.o + ((static_cast<int64_t>(u.b) * p.H + (valid ? h : 0)) * p.T + (valid ? pos : 0)) * D;
        const float4* odp = reinterpret_cast<const float4*>(scr + kUnitRows * 2) + row;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t os[32];
          tmem_ld32(o_tmem + c * 32, os);
          float od[32];
          if (p.S > 0 && valid) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 v4 = __ldcg(odp + (c * 8 + q4) * kUnitRows);
              od[4 * q4] = v4.x;
              od[4 * q4 + 1] = v4.y;
              od[4 * q4 + 2] = v4.z;
              od[4 * q4 + 3] = v4.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) od[i] = 0.f;
          }
          uint32_t pk2[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float x0 = __uint_as_float(os[i]) * ws + od[i] * wd;
            const float x1 = __uint_as_float(os[i + 1]) * ws + od[i + 1] * wd;
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
          p.lse[(static_cast<int64_t>(u.b) * p.H + h) * p.T + pos] = (m + __log2f(L)) * kLn2;
      }
      tc_fence_before();
      mbar_arrive(&o_free[t]);
      if (p.S > 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&dscr_empty[2 * slot + t]);
      }
    }
    if (!ok) raise_abort(abort_flag, p.status);
  } else {
    // ---------------------------------------------------------------- depth
    if (p.S > 0) {
      const int w = warp - 12;
      const uint8_t* ring_w = smem + C::OFF_DEP + w * p.nsw * p.dstage;
      uint8_t* pbuf = pbuf_base + w * (kMaxG * kMaxChunk * 2);
      uint64_t* dfull_w = dfull + w * kMaxNsw;
      // lanes per head: 32 / G rounded down to a power of two
      const int xl = p.G == 1 ? 32 : p.G == 2 ? 16 : p.G <= 4 ? 8 : 4;
      if (xl == 32)
        depth_warp_x<D, 32>(p, cta, n_c, w, lane, ring_w, dfull_w, dscr_full, dscr_empty, pbuf, scr_cta,
                            C::scratch_floats(), abort_flag);
      else if (xl == 16)
        depth_warp_x<D, 16>(p, cta, n_c, w, lane, ring_w, dfull_w, dscr_full, dscr_empty, pbuf, scr_cta,
                            C::scratch_floats(), abort_flag);
      else if (xl == 8)
        depth_warp_x<D, 8>(p, cta, n_c, w, lane, ring_w, dfull_w, dscr_full, dscr_empty, pbuf, scr_cta,
                           C::scratch_floats(), abort_flag);
      else
        depth_warp_x<D, 4>(p, cta, n_c, w, lane, ring_w, dfull_w, dscr_full, dscr_empty, pbuf, scr_cta,
                           C::scratch_floats(), abort_flag);
    }
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
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
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

// Q [B][H][T][D] bf16 as a 4-D tensor (D, T, H, B); box 64 x P x G x 1 (the head-major
// rows of one query tile); positions past T read as zeros.
bool make_q_map(CUtensorMap* map, const void* base, int D, int T, int H, int B, int P, int G) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2,
                                 static_cast<cuuint64_t>(H) * T * D * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(P), static_cast<cuuint32_t>(G), 1};
  return encode(map, base, 4, dims, strides, box);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

struct Plan {
  int P, n_pb, n_units, n_cta, sc, nck, nsw, dstage, smem;
};

// Depth streaming: every depth warp gets an equal share of the shared memory left after
// Q and the K/V ring, holding nsw (2..4) stages of one chunk of sc <= 32 slots (K and V)
// each; S is cut into the fewest chunks of equal size that allow two stages.
template <int D>
bool plan(const Problem& pr, Plan& pl) {
  using C = FwdCfg<D>;
  pl.P = BM / pr.G;
  pl.n_pb = (pr.T + 2 * pl.P - 1) / (2 * pl.P);
  pl.n_units = pr.B * pr.Hkv * pl.n_pb;
  const int sms = sm_count();
  if (sms <= 0) return false;
  pl.n_cta = std::min(pl.n_units, sms);
  if (pr.S == 0) {
    pl.sc = 1;
    pl.nck = 1;
    pl.nsw = 1;
    pl.dstage = 16;
  } else {
    const int per_warp = (kSmemLimit - C::smem_bytes(0)) / kDepthWarps;
    const int slot_pair = 2 * D * 2;  // one slot of K and of V
    // chunks of at most 32 slots, at least two stages per warp, as few chunks as possible
    const int cap = std::min(kMaxChunk, per_warp / (2 * slot_pair));
    if (cap <= 0) return false;
    pl.nck = (pr.S + cap - 1) / cap;
    pl.sc = (pr.S + pl.nck - 1) / pl.nck;
    pl.dstage = pl.sc * slot_pair;
    pl.nsw = std::min(kMaxNsw, per_warp / pl.dstage);
    if (pl.nsw < 2) return false;
  }
  pl.smem = C::smem_bytes(kDepthWarps * pl.nsw * pl.dstage);
  return pl.smem <= kSmemLimit;
}

template <int D>
cudaError_t launch(const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D>;
  const Problem& pr = a.p;
  Plan pl;
  if (!plan<D>(pr, pl)) return cudaErrorInvalidConfiguration;
  if (pr.S > 0 && (a.scratch == nullptr ||
                   a.scratch_bytes < static_cast<size_t>(pl.n_cta) * 2 * C::scratch_floats() * sizeof(float)))
    return cudaErrorInvalidValue;
  CUtensorMap tq, tk, tv;
  if (!make_q_map(&tq, a.q, D, pr.T, pr.H, pr.B, pl.P, pr.G) || !make_kv_map(&tk, a.k, D, pr.T, pr.B * pr.Hkv) ||
      !make_kv_map(&tv, a.v, D, pr.T, pr.B * pr.Hkv))
    return cudaErrorInvalidValue;
  FwdTcParams p;
  p.B = pr.B;
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.T = pr.T;
  p.S = pr.S;
  p.G = pr.G;
  p.P = pl.P;
  p.n_pb = pl.n_pb;
  p.n_units = pl.n_units;
  p.n_cta = pl.n_cta;
  p.sc = pl.sc;
  p.nck = pl.nck;
  p.nsw = pl.nsw;
  p.dstage = pl.dstage;
  p.scale_log2 = pr.scale_log2;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kd = static_cast<const __nv_bfloat16*>(a.kd);
  p.vd = static_cast<const __nv_bfloat16*>(a.vd);
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.scratch = static_cast<float*>(a.scratch);
  p.status = a.status;
  static int attr_bytes = 0;
  if (attr_bytes < pl.smem) {
    cudaError_t e = cudaFuncSetAttribute(moda_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
    if (e != cudaSuccess) return e;
    attr_bytes = pl.smem;
  }
  moda_fwd_tc_kernel<D><<<pl.n_cta, kThreads, pl.smem, s>>>(tq, tk, tv, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

bool fwd_sm103_supported(const Problem& p) {
  if (!((p.d == 64 || p.d == 128) && p.G >= 1 && p.G <= kMaxG && p.S <= kMaxS)) return false;
  if (sm_count() <= 0) return true;  // no device: argument checks only
  Plan pl;
  return p.d == 64 ? plan<64>(p, pl) : plan<128>(p, pl);
}

size_t fwd_sm103_workspace_bytes(const Problem& pr) {
  if (!fwd_sm103_supported(pr) || pr.S == 0) return 0;
  Plan pl;
  const bool ok = pr.d == 64 ? plan<64>(pr, pl) : plan<128>(pr, pl);
  if (!ok) return 0;
  const size_t per_cta = pr.d == 64 ? 2 * FwdCfg<64>::scratch_floats() : 2 * FwdCfg<128>::scratch_floats();
  return static_cast<size_t>(pl.n_cta) * per_cta * sizeof(float);
}

cudaError_t launch_fwd_sm103(const FwdArgs& a, cudaStream_t s) {
  return a.p.d == 64 ? launch<64>(a, s) : launch<128>(a, s);
}

}  // namespace moda
