// MoDA backward for bf16 on sm_103a.  The pages give no backward; these kernels
// evaluate the analytic gradient of the joint softmax (one denominator over the
// causal sequence keys and the same-position depth slots, "Mixture-of-Depths
// Attention", frame "One denominator allocates probability across both memories",
// Sec. 2.2 / Algorithm 1).  With P = exp(score - LSE), Delta_t = dO_t . O_t and
// dS = P (dO . value - Delta):
//
//   depth kernel (CUDA cores, warp per position):  dvd = sum_h P^d dO,
//       dkd = scale sum_h dS^d q, and the depth share of dq (scale sum_i dS^d kd_i),
//       kept in float32 in the workspace.
//   dK/dV kernel (tcgen05, one CTA per 128 keys of a kv head, looping over query tiles
//       of the G heads, 64 rows at d = 128, 128 at d = 64):  S^T = K Q^T, dP^T = V dO^T
//       into TMEM; thread k (TMEM lane k) forms P^T and dS^T, written back to TMEM as
//       bf16; dV += P^T dO, dK += dS^T Q with A read from TMEM.
//   dQ kernel (tcgen05, persistent: one CTA per SM walking blocks of 128 expanded query
//       rows, looping over key tiles of 64 at d = 128, 128 at d = 64):  S = Q K^T,
//       dP = dO V^T; thread r forms dS (bf16 into TMEM); dQ += dS K.  The epilogue adds
//       the depth share and rounds to bf16.
//
// All waits are bounded (see sm103_ptx.cuh); a timeout records MODA_ERR_TIMEOUT.
#include <cudaTypedefs.h>

#include <algorithm>

#include "moda_common.cuh"
#include "sm103_ptx.cuh"

namespace moda {
namespace {

using namespace sm103;

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  record_status(status, kStatusTimeout);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Key block and (b, kv head) of a dK/dV CTA.  CTAs run roughly in index order, so the
// index walks the (b, kv head) groups in bands of kKvBand: inside a band the smallest key
// blocks (most query tiles) come first, and the CTAs in flight at any time read the Q/dO
// rows of at most a band or two of groups, which stay in L2 between their reads (a
// group's Q and dO are read once by each of its key blocks).
constexpr int kKvBand = 8;
__device__ __forceinline__ void kv_block_of(int idx, int ngroups, int n_kblk, int& kblk, int& bg) {
  const int full = ngroups / kKvBand;  // complete bands
  if (idx < full * kKvBand * n_kblk) {
    const int band = idx / (kKvBand * n_kblk), r = idx % (kKvBand * n_kblk);
    kblk = r / kKvBand;
    bg = band * kKvBand + r % kKvBand;
  } else {
    const int rest = ngroups - full * kKvBand, r = idx - full * kKvBand * n_kblk;
    kblk = r / rest;
    bg = full * kKvBand + r % rest;
  }
}

struct BwdTcParams {
  int B, H, Hkv, T, S, G;
  int Tk;     // keys per (b, kv head) in k/v
  int delta;  // key j is visible to query position t iff j <= t + delta
  int S_read;  // slots read per position; dkd/dvd of slots S_read .. S-1 are written as zero
  float scale, scale_log2;
  const __nv_bfloat16 *q, *k, *v, *kd, *vd, *dout;
  const float* lse;
  float2* stats;  // {-lse * log2(e), Delta} per row (written by the depth kernel when S > 0)
  const __nv_bfloat16* o;  // forward output (Delta = dO . O)
  float* dq_accum;  // depth share of dq, float32 [B,H,T,d] (read by the dQ kernel when S > 0)
  __nv_bfloat16 *dq, *dk, *dv, *dkd, *dvd;
  float *dq_acc, *dk_acc, *dv_acc;  // set: dq/dk/dv are added to these in float32 instead
  int n_cta;  // CTAs of the persistent dQ kernel (d = 64)
  int* status;
};

// ============================================================================ depth
// One warp per position (b, g, t).  Lane = (slot sub-index j, 16-byte column chunk cc):
// a warp step covers SPW = 32 / (d/8) consecutive slots, each slot row read with one
// coalesced 16-byte copy per lane, staged by cp.async through a per-warp ring of
// kDepthStages steps in shared memory (seven steps in flight, no registers held; a lane
// only reads back the chunks it copied itself, so the group wait alone orders them).  The G heads of the position (HG >= G) stay in
// registers (q, dO packed bf16), so each depth element is read from HBM once and used
// for all G heads.  Each lane's partial dot products are summed over the slot's lanes by
// shuffles; with four heads a reduce-scatter hands every lane one full sum, so each
// head's P and dS are formed by two lanes and then gathered.  The warp also forms the row
// statistics of its G rows,
// {-lse * log2(e), Delta = dO . O}, and stores them for the dK/dV and dQ kernels.
constexpr int kDepthStages = 8;

template <int D, int HG>
__global__ void __launch_bounds__(256) moda_bwd_depth_kernel(const BwdTcParams p) {
  constexpr int CH = D / 8;
  constexpr int SPW = 32 / CH;
  constexpr int NB = kDepthStages;
  __shared__ __align__(16) uint4 stage[8][NB][2][32];  // [warp][step % NB][k, v][lane]
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t pid = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (pid >= static_cast<int64_t>(p.B) * p.Hkv * p.T) return;
  const int t = static_cast<int>(pid % p.T);
  const int64_t bg = pid / p.T;
  const int b = static_cast<int>(bg / p.Hkv), g = static_cast<int>(bg % p.Hkv);
  const int j = lane / CH, cc = lane % CH;

  const int64_t slab = pid * p.S * D;
  const int n_steps = (p.S_read + SPW - 1) / SPW;
  // copy step `st` (slots st*SPW + j) into ring entry st % NB; slots past S_read read as zero
  auto issue = [&](int st) {
    const int i = st * SPW + j;
    const bool sv = i < p.S_read;
    const int64_t off = sv ? slab + static_cast<int64_t>(i) * D + cc * 8 : 0;
    cp_async_16_zfill(smem_u32(&stage[wib][st % NB][0][lane]), p.kd + off, sv);
    cp_async_16_zfill(smem_u32(&stage[wib][st % NB][1][lane]), p.vd + off, sv);
  };
#pragma unroll
  for (int st = 0; st < NB - 1; ++st) {  // issued before the row loads
    if (st < n_steps) issue(st);
    cp_async_commit();
  }
  uint4 qv[HG], dv4[HG], ov[HG];
  float lse2[HG], dl[HG], dq[HG][8];
  int64_t rows[HG];
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {  // all row loads first, then the dependent arithmetic
    const bool hv = hh < p.G;
    rows[hh] = (static_cast<int64_t>(b) * p.H + g * p.G + (hv ? hh : 0)) * p.T + t;
    qv[hh] = hv ? __ldg(reinterpret_cast<const uint4*>(p.q + rows[hh] * D) + cc) : make_uint4(0, 0, 0, 0);
    dv4[hh] = hv ? __ldg(reinterpret_cast<const uint4*>(p.dout + rows[hh] * D) + cc) : make_uint4(0, 0, 0, 0);
    ov[hh] = hv ? __ldg(reinterpret_cast<const uint4*>(p.o + rows[hh] * D) + cc) : make_uint4(0, 0, 0, 0);
    lse2[hh] = hv ? __ldg(p.lse + rows[hh]) * kLog2e : INFINITY;
  }
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    float dsum = dot2_bf16(dv4[hh].x, ov[hh].x, 0.f);
    dsum = dot2_bf16(dv4[hh].y, ov[hh].y, dsum);
    dsum = dot2_bf16(dv4[hh].z, ov[hh].z, dsum);
    dsum = dot2_bf16(dv4[hh].w, ov[hh].w, dsum);
    dl[hh] = dsum;
  }
#pragma unroll
  for (int off = CH / 2; off >= 1; off >>= 1)
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) dl[hh] += __shfl_xor_sync(0xffffffffu, dl[hh], off);
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    if (hh < p.G && lane == 0) p.stats[rows[hh]] = make_float2(-lse2[hh], dl[hh]);
#pragma unroll
    for (int c = 0; c < 8; ++c) dq[hh][c] = 0.f;
  }
  // Four heads: the CH lanes of a slot hold 8 partial sums each (the scores and dP of the
  // four heads).  After plain butterfly steps down to groups of 8 lanes (d = 128), a
  // reduce-scatter leaves lane cc with the full sum number cc % 8 (head (cc % 8)/2; score
  // for even, dP for odd): at d = 64 7 shuffles instead of 24, at d = 128 15 instead of
  // 32; each head's P and dS are formed by its two lanes only, then gathered
  constexpr bool kScatter = CH >= 8 && HG == 4;
  float my_lse2 = 0.f, my_dl = 0.f;  // statistics of head (cc % 8)/2
  if constexpr (kScatter) {
    const int hm = (cc & 7) >> 1;
#pragma unroll
    for (int hh = 0; hh < HG; ++hh)
      if (hh == hm) {
        my_lse2 = lse2[hh];
        my_dl = dl[hh];
      }
  }
  for (int st = 0; st < n_steps; ++st) {
    const int i = st * SPW + j;
    const bool sv = i < p.S_read;
    if (st + NB - 1 < n_steps) issue(st + NB - 1);
    cp_async_commit();
    cp_async_wait<NB - 1>();  // this thread's copies of step st have landed
    const uint4 kv = stage[wib][st % NB][0][lane], vv = stage[wib][st % NB][1][lane];
    float s[HG], dp[HG];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      float a = 0.f, c2 = 0.f;
      a = dot2_bf16(qv[hh].x, kv.x, a);
      a = dot2_bf16(qv[hh].y, kv.y, a);
      a = dot2_bf16(qv[hh].z, kv.z, a);
      a = dot2_bf16(qv[hh].w, kv.w, a);
      c2 = dot2_bf16(dv4[hh].x, vv.x, c2);
      c2 = dot2_bf16(dv4[hh].y, vv.y, c2);
      c2 = dot2_bf16(dv4[hh].z, vv.z, c2);
      c2 = dot2_bf16(dv4[hh].w, vv.w, c2);
      s[hh] = a;
      dp[hh] = c2;
    }
    // P and dS enter the gradient products rounded to bf16, as in the tensor-core kernels,
    // so every product is a mixed-precision FMA on the stored bf16 pairs (no widening)
    uint32_t pdv[HG];  // per head: P in the low half, dS in the high half
    if constexpr (kScatter) {
      float v[8];
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        v[2 * hh] = s[hh];
        v[2 * hh + 1] = dp[hh];
      }
#pragma unroll
      for (int off = CH / 2; off >= 8; off >>= 1)
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] += __shfl_xor_sync(0xffffffffu, v[u], off);
      // reduce-scatter over 8 lanes: keep the half named by each low bit of cc
      const bool b2 = (cc & 4) != 0, b1 = (cc & 2) != 0, b0 = (cc & 1) != 0;
      float w4[4], w2[2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float send = b2 ? v[u] : v[u + 4];
        w4[u] = (b2 ? v[u + 4] : v[u]) + __shfl_xor_sync(0xffffffffu, send, 4);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float send = b1 ? w4[u] : w4[u + 2];
        w2[u] = (b1 ? w4[u + 2] : w4[u]) + __shfl_xor_sync(0xffffffffu, send, 2);
      }
      const float mine = (b0 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b0 ? w2[0] : w2[1], 1);
      const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
      const float sc = b0 ? other : mine, dpp = b0 ? mine : other;
      const float pr = sv ? ex2(fmaf(sc, p.scale_log2, -my_lse2)) : 0.f;
      const uint32_t pd = pack_bf16(pr, pr * (dpp - my_dl));
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) pdv[hh] = __shfl_sync(0xffffffffu, pd, (lane & ~(CH - 1)) | (2 * hh));
    } else {
      // full dot products: reduce over the CH lanes of this slot
#pragma unroll
      for (int off = CH / 2; off >= 1; off >>= 1) {
#pragma unroll
        for (int hh = 0; hh < HG; ++hh) {
          s[hh] += __shfl_xor_sync(0xffffffffu, s[hh], off);
          dp[hh] += __shfl_xor_sync(0xffffffffu, dp[hh], off);
        }
      }
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        const float pr = sv ? ex2(fmaf(s[hh], p.scale_log2, -lse2[hh])) : 0.f;
        pdv[hh] = pack_bf16(pr, pr * (dp[hh] - dl[hh]));
      }
    }
    const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
    float gk[8], gv[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) gk[c] = gv[c] = 0.f;
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      const uint32_t pd = pdv[hh];
      const uint32_t qw[4] = {qv[hh].x, qv[hh].y, qv[hh].z, qv[hh].w};
      const uint32_t ow[4] = {dv4[hh].x, dv4[hh].y, dv4[hh].z, dv4[hh].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        axpy2_bf16_hi(pd, qw[c], gk[2 * c], gk[2 * c + 1]);
        axpy2_bf16(pd, ow[c], gv[2 * c], gv[2 * c + 1]);
        axpy2_bf16_hi(pd, kw[c], dq[hh][2 * c], dq[hh][2 * c + 1]);
      }
    }
    if (sv) {
      uint4 ok, ov;
      ok.x = pack_bf16(gk[0] * p.scale, gk[1] * p.scale);
      ok.y = pack_bf16(gk[2] * p.scale, gk[3] * p.scale);
      ok.z = pack_bf16(gk[4] * p.scale, gk[5] * p.scale);
      ok.w = pack_bf16(gk[6] * p.scale, gk[7] * p.scale);
      ov.x = pack_bf16(gv[0], gv[1]);
      ov.y = pack_bf16(gv[2], gv[3]);
      ov.z = pack_bf16(gv[4], gv[5]);
      ov.w = pack_bf16(gv[6], gv[7]);
      reinterpret_cast<uint4*>(p.dkd + slab + static_cast<int64_t>(i) * D)[cc] = ok;
      reinterpret_cast<uint4*>(p.dvd + slab + static_cast<int64_t>(i) * D)[cc] = ov;
    }
  }
  // slots in memory that are not read have zero gradient
  for (int i = p.S_read + j; i < p.S; i += SPW) {
    reinterpret_cast<uint4*>(p.dkd + slab + static_cast<int64_t>(i) * D)[cc] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(p.dvd + slab + static_cast<int64_t>(i) * D)[cc] = make_uint4(0, 0, 0, 0);
  }
  // dq depth share: sum over the SPW slot groups and write float32
  if constexpr (kScatter) {
    // reduce-scatter over the groups: group j ends with the full sums of heads
    // j*(4/SPW) .. j*(4/SPW) + 4/SPW - 1, and writes them
    constexpr int NV = HG * 8;
    float val[NV];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh)
#pragma unroll
      for (int c = 0; c < 8; ++c) val[hh * 8 + c] = dq[hh][c];
    int n = NV;
#pragma unroll
    for (int off = 16; off >= CH; off >>= 1) {
      const bool bit = (lane & off) != 0;
      n >>= 1;
#pragma unroll
      for (int u = 0; u < NV / 2; ++u) {
        if (u < n) {
          const float send = bit ? val[u] : val[u + n];
          val[u] = (bit ? val[u + n] : val[u]) + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
    }
    constexpr int NH = 4 / SPW;  // heads per group
#pragma unroll
    for (int u = 0; u < NH; ++u) {
      const int hh = j * NH + u;
      if (hh < p.G) {
        const int64_t row = (static_cast<int64_t>(b) * p.H + g * p.G + hh) * p.T + t;
        float4* dst = reinterpret_cast<float4*>(p.dq_accum + row * D + cc * 8);
        const float* w = val + u * 8;
        dst[0] = make_float4(w[0] * p.scale, w[1] * p.scale, w[2] * p.scale, w[3] * p.scale);
        dst[1] = make_float4(w[4] * p.scale, w[5] * p.scale, w[6] * p.scale, w[7] * p.scale);
      }
    }
  } else {
#pragma unroll
    for (int off = CH; off < 32; off <<= 1) {
#pragma unroll
      for (int hh = 0; hh < HG; ++hh)
#pragma unroll
        for (int c = 0; c < 8; ++c) dq[hh][c] += __shfl_xor_sync(0xffffffffu, dq[hh][c], off);
    }
    if (j == 0) {
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        if (hh < p.G) {
          const int64_t row = (static_cast<int64_t>(b) * p.H + g * p.G + hh) * p.T + t;
          float4* dst = reinterpret_cast<float4*>(p.dq_accum + row * D + cc * 8);
          dst[0] = make_float4(dq[hh][0] * p.scale, dq[hh][1] * p.scale, dq[hh][2] * p.scale, dq[hh][3] * p.scale);
          dst[1] = make_float4(dq[hh][4] * p.scale, dq[hh][5] * p.scale, dq[hh][6] * p.scale, dq[hh][7] * p.scale);
        }
      }
    }
  }
}

// Row blocks of the persistent dQ kernels: block index i -> (position block, b, kv head), the
// longest rows first; CTA c takes blocks c, 2C-1-c, 2C+c, ... (snake order over C CTAs), so
// that every CTA gets a similar amount of work.
__device__ __forceinline__ int dq_blocks_of_cta(int n_blocks, int n_cta, int c) {
  const int R = n_blocks / n_cta, rem = n_blocks % n_cta;
  const bool extra = (R & 1) ? (n_cta - 1 - c < rem) : (c < rem);
  return R + (extra ? 1 : 0);
}

struct DqBlock {
  int b, g, bg, p0, n_kv;
};

__device__ __forceinline__ DqBlock dq_block_at(const BwdTcParams& p, int P, int c, int k, int tile_keys) {
  const int idx = k * p.n_cta + ((k & 1) ? p.n_cta - 1 - c : c);
  const int ngroups = p.B * p.Hkv;
  const int n_pb = (p.T + P - 1) / P;
  DqBlock x;
  x.bg = idx % ngroups;
  x.b = x.bg / p.Hkv;
  x.g = x.bg % p.Hkv;
  x.p0 = (n_pb - 1 - idx / ngroups) * P;
  const int p_last = min(x.p0 + P, p.T) - 1;
  x.n_kv = min((p_last + p.delta) / tile_keys + 1, (p.Tk + tile_keys - 1) / tile_keys);
  return x;
}

// ============================================================================ dQ
// Persistent CTAs (one per SM) walking row blocks of 128 expanded rows of (b, g),
// position-major (row r -> position p0 + r/G, head g*G + r%G), P = floor(128/G) positions.
// Keys in tiles of 64.  Used at d = 128 (d = 64 has a kernel of its own below).  A block's
// Q and dO are staged by TMA and copied into TMEM by warpgroup 0 right after the previous
// block's last tile; the K/V ring runs on across blocks.
// Warps: 0 TMA (K_j and V_j in one transaction), 1 TMEM and the S/dP products, 2 ..
// 2+4*NWG-1 gradient warps (warp w owns TMEM lanes 32*(w%4) ..; with two warpgroups WG k
// handles key columns [32k, 32k+32) of every tile, with one it handles all 64; WG 0 also
// writes the CTA's Q and dO rows into TMEM), 2+4*NWG the dQ products.  NBUF S/dP buffers:
// with 2 the tensor cores compute tile j+1 while tile j's dS is formed.
// TMEM: S[b] cols [64b, 64b+64), dP[b] [64(NBUF+b), ...), dQ [128 NBUF, 128 NBUF + d),
// then Q and dO (bf16 pairs, d/2 columns each: the A operands of S and dP).  dS (bf16)
// is written over S[b]: warpgroup w packs its 32 keys into the first 16 columns of its own
// half [32w, 32w+32) (packed_col below), so no warpgroup overwrites columns another still reads.
constexpr int QBM = 128, QBN = 64;

// TMEM column (from the start of a 64-column S or dP buffer) of the bf16 pairs of keys (or
// queries) 16kk .. 16kk+15, the A operand of step kk of a 64-deep gradient product.  With two
// warpgroups splitting a buffer's 64 columns, warpgroup w packs its 32 values into the first
// 16 columns of its own half [32w, 32w+32): columns the other warpgroup still reads are never
// written.
template <int NWG>
__device__ __forceinline__ uint32_t packed_col(int kk) {
  return NWG == 2 ? static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8) : static_cast<uint32_t>(kk * 8);
}

template <int D, int NBUF, int NWG>
struct DqCfg {
  static constexpr int THREADS = 64 + 128 * NWG + 32;  // + the dQ-issuing warp
  static constexpr int KV_BYTES = QBN * D * 2;  // one K (or V) tile; a ring slot holds both
  static constexpr int NSLOT = 4;
  static constexpr int OFF_KV = 0;
  // Q and dO of a block staged by TMA (64-column halves, 128-byte swizzle) on their way into TMEM
  static constexpr int QS_HALF = QBM * 128;
  static constexpr int OFF_QS = OFF_KV + NSLOT * 2 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_QS + 2 * (D / 64) * QS_HALF;
  // kv_full[NSLOT], kv_empty[NSLOT], q_full, s_full[NBUF], ds_full[NBUF], drain, last_done,
  // qs_full, qs_empty, drain_dq
  static constexpr int NBAR = 2 * NSLOT + 6 + 2 * NBUF;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  // Q and dO of the CTA's rows (bf16 pairs, D/2 columns each) are the A operands of S, dP
  static constexpr uint32_t TM_S = 0, TM_DP = 64 * NBUF, TM_DQ = 128 * NBUF, TM_Q = TM_DQ + D, TM_DO = TM_Q + D / 2;
  static constexpr uint32_t TM_COLS = (TM_DO + D / 2) <= 256 ? 256 : 512;
  static_assert(TM_DO + D / 2 <= 512, "TMEM columns");
  // a CTA that takes all 512 columns must be alone on its SM: shared memory keeps a second out
  static_assert(TM_COLS < 512 || SMEM > 116 * 1024, "one CTA per SM");
};

template <int D, int NBUF, int NWG>
__global__ void __launch_bounds__(DqCfg<D, NBUF, NWG>::THREADS, NBUF == 1 ? 2 : 1)
    moda_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                       const BwdTcParams p) {
  using C = DqCfg<D, NBUF, NWG>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = QBM / p.G;
  const int cta = static_cast<int>(blockIdx.x);
  const int n_blk = dq_blocks_of_cta((p.T + P - 1) / P * p.B * p.Hkv, p.n_cta, cta);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::NSLOT;
  uint64_t* q_full = bars + 2 * C::NSLOT;
  uint64_t* s_full = q_full + 1;
  uint64_t* ds_full = s_full + NBUF;
  uint64_t* drain = ds_full + NBUF;
  uint64_t* last_done = drain + 1;
  uint64_t* qs_full = last_done + 1;   // a block's Q and dO staged in shared memory
  uint64_t* qs_empty = qs_full + 1;    // ... and copied from there into TMEM
  uint64_t* drain_dq = qs_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(q_full, 128);
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&ds_full[i], 128 * NWG);
    }
    mbar_init(drain, 1);
    mbar_init(drain_dq, 1);
    mbar_init(last_done, 1);
    mbar_init(qs_full, 1);
    mbar_init(qs_empty, 128);  // warpgroup 0 of the gradient warps
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Barrier phases, ring slots and S/dP buffers follow the running count of key tiles over
  // the CTA's row blocks; q_full, qs_full/qs_empty and last_done follow the block count.
  if (warp == 0) {
    // ---------------------------------------------------------------- Q/dO staging, K_j, V_j loads
    if (lane == 0) {
      int it = 0, staged = 0;
      bool ok = true;
      for (int k = 0; ok && k < n_blk; ++k) {
        const DqBlock x = dq_block_at(p, P, cta, k, QBN);
        // this block's Q and dO rows (position-major; positions past T read as zeros), once
        // the previous block's have been copied out of the staging buffer
        if (k > 0 && !mbar_wait(qs_empty, (k - 1) & 1, abort_flag)) {
          raise_abort(abort_flag, p.status);
          break;
        }
        mbar_arrive_expect_tx(qs_full, 2u * (D / 64) * p.G * P * 128u);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(smem + C::OFF_QS + h * C::QS_HALF, &tmQ, qs_full, h * 64, x.g * p.G, x.p0, x.b);
          tma_load_4d(smem + C::OFF_QS + (D / 64 + h) * C::QS_HALF, &tmO, qs_full, h * 64, x.g * p.G, x.p0, x.b);
        }
        staged = k + 1;
        for (int j = 0; j < x.n_kv; ++j, ++it) {
          const int slot = it % C::NSLOT, use = it / C::NSLOT;
          if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, abort_flag)) {
            raise_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::OFF_KV + slot * 2 * C::KV_BYTES;
          mbar_arrive_expect_tx(&kv_full[slot], 2 * C::KV_BYTES);
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_3d(dst + h * (QBN * 128), &tmK, &kv_full[slot], h * 64, j * QBN, x.bg);
            tma_load_3d(dst + C::KV_BYTES + h * (QBN * 128), &tmV, &kv_full[slot], h * 64, j * QBN, x.bg);
          }
        }
      }
      if (*abort_flag) {
        volatile int never = 0;
        for (int j = max(0, it - C::NSLOT); j < it; ++j) mbar_wait(&kv_full[j % C::NSLOT], (j / C::NSLOT) & 1, &never);
        if (staged > 0) mbar_wait(qs_full, (staged - 1) & 1, &never);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- S, dP issuer
    // S and dP of tile t go to buffer t % NBUF, over the dS of tile t - NBUF: issued once the
    // dQ product of that tile has completed (its commit completes that tile's phase of
    // kv_empty).  The first tile of a block waits for the block's Q and dO in TMEM.
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(QBM, QBN, false);
      // descriptors built once; each MMA only advances the start address
      const uint64_t kv_desc_k = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);            // K-major
      bool ok = true;
      int t = 0;
      for (int k = 0; ok && k < n_blk; ++k) {
        const int n_kv = dq_block_at(p, P, cta, k, QBN).n_kv;
        ok = mbar_wait(q_full, k & 1, abort_flag);
        for (int j = 0; ok && j < n_kv; ++j, ++t) {
          const int slot = t % C::NSLOT, bf = t % NBUF;
          ok = mbar_wait(&kv_full[slot], (t / C::NSLOT) & 1, abort_flag) &&
               (t < NBUF || mbar_wait(&kv_empty[(t - NBUF) % C::NSLOT], ((t - NBUF) / C::NSLOT) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          const uint64_t k_desc = sdesc_add(kv_desc_k, slot * 2 * C::KV_BYTES);
          const uint64_t v_desc = sdesc_add(k_desc, C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t boff = (kk >> 2) * (QBN * 128) + (kk & 3) * 32;
            mma_bf16_ts(tmem + C::TM_S + bf * QBN, tmem + C::TM_Q + kk * 8, sdesc_add(k_desc, boff), IDESC_S, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t boff = (kk >> 2) * (QBN * 128) + (kk & 3) * 32;
            mma_bf16_ts(tmem + C::TM_DP + bf * QBN, tmem + C::TM_DO + kk * 8, sdesc_add(v_desc, boff), IDESC_S,
                        kk > 0);
          }
          mma_commit(&s_full[bf]);
        }
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
      }
    }
  } else if (warp == 2 + 4 * NWG) {
    // ---------------------------------------------------------------- dQ issuer
    // dQ of tile t follows ds_full(t), which the gradient warps signal only after reading
    // S(t), dP(t): those MMAs have completed, so this thread's commit after dQ(t) is the last
    // use of K_t, V_t and of the buffer's dS, and frees both.  The first dQ of a block
    // overwrites the accumulator: the gradient warps signal its ds_full only after their
    // epilogue of the previous block has read it.
    if (lane == 0) {
      constexpr uint32_t IDESC_DQ = idesc_bf16(QBM, D, true);
      const uint64_t kv_desc_mn = sdesc_sw128(sbase + C::OFF_KV, QBN * 128, 1024);    // MN-major
      bool ok = true;
      int t = 0;
      for (int k = 0; ok && k < n_blk; ++k) {
        const int n_kv = dq_block_at(p, P, cta, k, QBN).n_kv;
        for (int j = 0; ok && j < n_kv; ++j, ++t) {
          const int slot = t % C::NSLOT, bf = t % NBUF;
          ok = mbar_wait(&ds_full[bf], (t / NBUF) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t k_desc = sdesc_add(kv_desc_mn, slot * 2 * C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < QBN / 16; ++kk)
            mma_bf16_ts(tmem + C::TM_DQ, tmem + C::TM_S + bf * QBN + packed_col<NWG>(kk),
                        sdesc_add(k_desc, kk * 16 * 128), IDESC_DQ, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&kv_empty[slot]);  // K_t, V_t and the buffer's dS no longer read
        }
        if (ok) mma_commit(last_done);  // this block's dQ is complete
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        mma_commit(drain_dq);
        volatile int never = 0;
        mbar_wait(drain_dq, 0, &never);
      }
    }
  } else {
    // ---------------------------------------------------------------- gradients (thread = row)
    const int wg = (warp - 2) >> 2;
    constexpr int NCOL = QBN / NWG;  // key columns of a tile this warpgroup forms
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool row_in = r < P * p.G;
    // row r of Q and dO of block k into TMEM lane r: column c holds elements 2c, 2c+1, the
    // row's 32-bit words as stored.  The rows come from the staging buffer (per 64-column
    // half, row r: 128 bytes, 16-byte chunk c at chunk c ^ (r % 8)); rows past P*G, which the
    // TMA box does not cover, are zero.
    auto load_q = [&](int k) -> bool {
      if (!warp_wait(qs_full, k & 1, abort_flag)) return false;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          const uint32_t src = sbase + C::OFF_QS + (part * (D / 64) + h) * C::QS_HALF + r * 128;
          uint32_t w[32];
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 a = row_in ? ld_shared_v4(src + ((ch ^ (r & 7)) << 4)) : make_uint4(0, 0, 0, 0);
            w[4 * ch] = a.x;
            w[4 * ch + 1] = a.y;
            w[4 * ch + 2] = a.z;
            w[4 * ch + 3] = a.w;
          }
          tmem_st32_nowait(tmem + lane_base + (part ? C::TM_DO : C::TM_Q) + h * 32, w);
        }
      }
      mbar_arrive(qs_empty);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_full);
      return true;
    };
    auto row_of = [&](int k, bool& valid) -> int64_t {
      const DqBlock x = dq_block_at(p, P, cta, k, QBN);
      const int pos = x.p0 + r / p.G;
      valid = row_in && pos < p.T;
      return (static_cast<int64_t>(x.b) * p.H + x.g * p.G + r % p.G) * p.T + (valid ? pos : 0);
    };
    bool ok = !(wg == 0 && n_blk > 0) || load_q(0);
    const float sl2 = p.scale_log2;
    float2 stt_next = make_float2(-INFINITY, 0.f);  // row statistics of the next block
    if (n_blk > 0) {
      bool v0;
      const int64_t r0 = row_of(0, v0);
      if (v0) stt_next = p.stats[r0];
    }
    int t = 0;
    for (int k = 0; ok && k < n_blk; ++k) {
      const DqBlock x = dq_block_at(p, P, cta, k, QBN);
      const int pos = x.p0 + r / p.G;
      const bool valid = row_in && pos < p.T;
      const int h = x.g * p.G + r % p.G;
      const int64_t row = (static_cast<int64_t>(x.b) * p.H + h) * p.T + (valid ? pos : 0);
      const float nlse2 = stt_next.x;  // -lse * log2(e)
      const float dlt = stt_next.y;
      // the depth share this thread adds in the epilogue into L2 now
      if (p.S > 0 && valid) {
#pragma unroll
        for (int c0 = wg * (D / NWG); c0 < (wg + 1) * (D / NWG); c0 += 32) prefetch_l2(p.dq_accum + row * D + c0);
      }
      const int key_end = min(pos + p.delta, p.Tk - 1);  // last key this row sees
      for (int j = 0; j < x.n_kv; ++j, ++t) {
        const int bf = t % NBUF;
        ok = warp_wait(&s_full[bf], (t / NBUF) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        uint32_t pk[NCOL / 2];
#pragma unroll
        for (int hf = 0; hf < NCOL / 32; ++hf) {
          const int c0 = wg * NCOL + hf * 32;  // first key column of this group
          uint32_t s[32], dpv[32];
          tmem_ld32x2(tmem + lane_base + C::TM_S + bf * QBN + c0, tmem + lane_base + C::TM_DP + bf * QBN + c0, s, dpv);
          const int lim = valid ? key_end - (j * QBN + c0) : -1;  // columns c <= lim are visible
          float e[32];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            ffma2(__uint_as_float(s[c]), __uint_as_float(s[c + 1]), sl2, sl2, nlse2, nlse2, e[c], e[c + 1]);
            e[c] = ex2(e[c]);
            e[c + 1] = ex2(e[c + 1]);
          }
          if (lim < 31) {
#pragma unroll
            for (int c = 0; c < 32; ++c) e[c] = (c <= lim) ? e[c] : 0.f;
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float d0, d1;
            fsubmul2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1]), dlt, dlt, e[c], e[c + 1], d0, d1);
            pk[hf * 16 + (c >> 1)] = pack_bf16(d0, d1);
          }
        }
        // dS (bf16 pairs) over this warpgroup's own S columns of S[bf] (see packed_col)
        if constexpr (NCOL == 64)
          tmem_st32(tmem + lane_base + C::TM_S + bf * QBN, pk);
        else
          tmem_st16(tmem + lane_base + C::TM_S + bf * QBN + wg * 32, pk);
        tc_fence_before();
        mbar_arrive(&ds_full[bf]);
      }
      if (!ok) break;
      // the S and dP products of this block have completed (their results were read): Q and
      // dO of the next block replace theirs first, so that the next block's products can
      // start while this block's epilogue runs
      if (wg == 0 && k + 1 < n_blk && !load_q(k + 1)) {
        ok = false;
        break;
      }
      if (k + 1 < n_blk) {
        bool vn;
        const int64_t rn = row_of(k + 1, vn);
        stt_next = vn ? p.stats[rn] : make_float2(-INFINITY, 0.f);
      }
      ok = warp_wait(last_done, k & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      // WG w writes dq columns [w*D/NWG, (w+1)*D/NWG)
#pragma unroll 1
      for (int c0 = wg * (D / NWG); c0 < (wg + 1) * (D / NWG); c0 += 32) {
        uint32_t acc[32];
        tmem_ld32(tmem + lane_base + C::TM_DQ + c0, acc);
        float extra[32];
        if (p.S > 0 && valid) {
          const float4* src = reinterpret_cast<const float4*>(p.dq_accum + row * D + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 e = src[i];
            extra[4 * i] = e.x;
            extra[4 * i + 1] = e.y;
            extra[4 * i + 2] = e.z;
            extra[4 * i + 3] = e.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) extra[i] = 0.f;
        }
        if (valid && p.dq_acc != nullptr) {
          float4* dst = reinterpret_cast<float4*>(p.dq_acc + row * D + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 y = dst[i];
            y.x += fmaf(__uint_as_float(acc[4 * i]), p.scale, extra[4 * i]);
            y.y += fmaf(__uint_as_float(acc[4 * i + 1]), p.scale, extra[4 * i + 1]);
            y.z += fmaf(__uint_as_float(acc[4 * i + 2]), p.scale, extra[4 * i + 2]);
            y.w += fmaf(__uint_as_float(acc[4 * i + 3]), p.scale, extra[4 * i + 3]);
            dst[i] = y;
          }
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.dq + row * D + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              const int c = 8 * i + 2 * k2;
              w[k2] = pack_bf16(fmaf(__uint_as_float(acc[c]), p.scale, extra[c]),
                                fmaf(__uint_as_float(acc[c + 1]), p.scale, extra[c + 1]));
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      // the accumulator read is complete (tcgen05.ld waits) before this warp's next ds_full
      tc_fence_before();
    }
    if (!ok) raise_abort(abort_flag, p.status);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ============================================================================ dK / dV
// CTA: 128 keys [kb, kb+128) of (b, g).  Query tiles of 64 rows, head-major inside the
// tile (row r -> head g*G + r/P', position p0 + r%P', P' = floor(64/G)), loaded by TMA
// together with dO; their LSE and Delta are copied asynchronously by the producer warp.
// Warps: 0 loads, 1 TMEM and the S^T/dP^T products, 2 .. 2+4*NWG-1 gradient warps
// (thread = key = TMEM lane; with two warpgroups WG k handles query columns [32k, 32k+32),
// with one all 64), 2+4*NWG the dV and 3+4*NWG the dK products: three issuing threads, so
// that one waiting on a barrier leaves the others' MMAs running, and the N = 64 products
// are not issued by one thread alone.
// TMEM: S^T[b] cols [64b, ..), dP^T[b] [64(NBUF+b), ..), dV [128 NBUF, +d), dK [+d, +2d).
// P^T and dS^T (bf16) are written over their buffers the same way as dS in the dQ kernel
// (packed_col): warpgroup w's 32 query columns into the first 16 columns of its own half.
constexpr int KBM = 128, KBN = 64;

template <int D, int NBUF, int NWG>
struct DkvCfg {
  static constexpr int THREADS = 64 + 128 * NWG + 64;  // + the dV and dK issuing warps
  static constexpr int KV_BYTES = KBM * D * 2;   // the CTA's K (or V) tile
  static constexpr int QT_BYTES = KBN * D * 2;   // one 64-row Q (or dO) tile
  static constexpr int NSTAGE = 4;
  static constexpr int STAGE_BYTES = 2 * QT_BYTES;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_BYTES;
  static constexpr int OFF_Q = 2 * KV_BYTES;     // stage s: Q at + s*STAGE, dO at + QT_BYTES
  static constexpr int OFF_STAT = OFF_Q + NSTAGE * STAGE_BYTES;  // [NSTAGE][64] {-lse*log2e, Delta}
  static constexpr int OFF_BAR = OFF_STAT + NSTAGE * 2 * KBN * 4;
  // kv_full, q_full[NSTAGE], q_empty[NSTAGE], s_full[NBUF], p_full[NBUF], drain, last_done,
  // dp_full[NBUF] (S^T and dP^T of a buffer complete separately), drain_g[2]
  static constexpr int NBAR = 5 + 2 * NSTAGE + 3 * NBUF;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr uint32_t TM_S = 0, TM_DP = 64 * NBUF, TM_DV = 128 * NBUF, TM_DK = 128 * NBUF + D;
  static constexpr uint32_t TM_COLS = (TM_DK + D) <= 256 ? 256 : 512;
};

template <int D, int NBUF, int NWG>
__global__ void __launch_bounds__(DkvCfg<D, NBUF, NWG>::THREADS, NBUF == 1 ? 2 : 1)
    moda_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                         const BwdTcParams p) {
  using C = DkvCfg<D, NBUF, NWG>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Pq = KBN / p.G;  // positions per query tile
  const int ngroups = p.B * p.Hkv;
  int kblk, bg;
  kv_block_of(static_cast<int>(blockIdx.x), ngroups, (p.Tk + KBM - 1) / KBM, kblk, bg);
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int kb = kblk * KBM;
  // first query tile whose rows see key kb: position kb - delta (every key of the range is
  // seen by position T - 1, so qt0 <= qt1)
  const int qt0 = max(kb - p.delta, 0) / Pq, qt1 = (p.T - 1) / Pq;
  const int n_q = qt1 - qt0 + 1;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + C::NSTAGE;
  uint64_t* s_full = q_empty + C::NSTAGE;
  uint64_t* p_full = s_full + NBUF;
  uint64_t* drain = p_full + NBUF;
  uint64_t* last_done = drain + 1;
  uint64_t* dp_full = last_done + 1;
  uint64_t* drain_g = dp_full + NBUF;  // [2]: the dV and the dK issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const float4* stat = reinterpret_cast<const float4*>(smem + C::OFF_STAT);  // two rows per float4

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(&q_full[i], 1 + 32);  // TMA arrive + one cp.async arrival per producer lane
      mbar_init(&q_empty[i], 2);  // the dV and the dK issuer
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&dp_full[i], 1);
      mbar_init(&p_full[i], 128 * NWG);
    }
    mbar_init(drain, 1);
    mbar_init(&drain_g[0], 1);
    mbar_init(&drain_g[1], 1);
    mbar_init(last_done, 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // rows past Pq*G of every query tile are never written by TMA: zero them once
  if (Pq * p.G < KBN) {
    for (int i = threadIdx.x; i < C::NSTAGE * C::STAGE_BYTES / 16; i += blockDim.x)
      st_shared_v4(sbase + C::OFF_Q + i * 16, make_uint4(0, 0, 0, 0));
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmO);
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
    // ---------------------------------------------------------------- loads
    bool ok = true;
    int issued = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        tma_load_3d(smem + C::OFF_K + h * (KBM * 128), &tmK, kv_full, h * 64, kb, bg);
        tma_load_3d(smem + C::OFF_V + h * (KBM * 128), &tmV, kv_full, h * 64, kb, bg);
      }
    }
    for (int i = 0; i < n_q; ++i) {
      const int st = i % C::NSTAGE, use = i / C::NSTAGE;
      if (use > 0 && !warp_wait(&q_empty[st], (use - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const int p0 = (qt0 + i) * Pq;
      // row statistics (LSE, Delta) of this tile, copied asynchronously.  Rows that do not
      // exist (head >= G or position >= T) read a valid row's statistics: their Q and dO rows
      // are zero in shared memory, so whatever finite P and dS they get contributes nothing.
      const uint32_t sl = sbase + C::OFF_STAT + st * KBN * 8;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int r = lane + 32 * rr;
        const int hh = min(r / Pq, p.G - 1), pos = min(p0 + r % Pq, p.T - 1);
        const int64_t row = (static_cast<int64_t>(b) * p.H + g * p.G + hh) * p.T + pos;
        cp_async_8(sl + r * 8, p.stats + row);
      }
      cp_async_arrive_noinc(&q_full[st]);
      if (lane == 0) {
        uint8_t* dst = smem + C::OFF_Q + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&q_full[st], static_cast<uint32_t>(2 * Pq * p.G * D * 2));
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(dst + h * (KBN * 128), &tmQ, &q_full[st], h * 64, p0, b * p.H + g * p.G);
          tma_load_3d(dst + C::QT_BYTES + h * (KBN * 128), &tmO, &q_full[st], h * 64, p0, b * p.H + g * p.G);
        }
      }
      issued = i + 1;
    }
    if (!ok || *abort_flag) {
      if (lane == 0) {
        raise_abort(abort_flag, p.status);
        volatile int never = 0;
        mbar_wait(kv_full, 0, &never);
      }
      volatile int never = 0;
      for (int i = max(0, issued - C::NSTAGE); i < issued; ++i)
        mbar_wait(&q_full[i % C::NSTAGE], (i / C::NSTAGE) & 1, &never);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- S^T, dP^T issuer
    // S^T and dP^T of tile i go to buffer i % NBUF, over the P^T and dS^T of tile i - NBUF:
    // issued once the dV and dK products of that tile have completed (they commit q_empty)
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(KBM, KBN, false);
      // descriptors built once; each MMA only advances the start address
      const uint64_t k_desc = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
      const uint64_t qt_desc_k = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);           // K-major Q/dO tiles
      bool ok = mbar_wait(kv_full, 0, abort_flag);
      for (int i = 0; ok && i < n_q; ++i) {
        const int st = i % C::NSTAGE, bf = i % NBUF;
        ok = mbar_wait(&q_full[st], (i / C::NSTAGE) & 1, abort_flag) &&
             (i < NBUF || mbar_wait(&q_empty[(i - NBUF) % C::NSTAGE], ((i - NBUF) / C::NSTAGE) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint64_t q_desc = sdesc_add(qt_desc_k, st * C::STAGE_BYTES);
        const uint64_t o_desc = sdesc_add(q_desc, C::QT_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * (KBM * 128) + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * (KBN * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + C::TM_S + bf * KBN, sdesc_add(k_desc, aoff), sdesc_add(q_desc, boff), IDESC_S, kk > 0);
        }
        mma_commit(&s_full[bf]);  // the gradient warps form P^T while dP^T is computed
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * (KBM * 128) + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * (KBN * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + C::TM_DP + bf * KBN, sdesc_add(v_desc, aoff), sdesc_add(o_desc, boff), IDESC_S, kk > 0);
        }
        mma_commit(&dp_full[bf]);
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
      }
    }
  } else if (warp >= 2 + 4 * NWG) {
    // ---------------------------------------------------------------- dV (first), dK (second) issuers
    // dV, dK of tile i follow p_full(i): the gradient warps have read S^T(i), dP^T(i) and
    // written P^T, dS^T over them.  Each thread's commit after its product is its share of
    // the release of the Q/dO stage and of the buffer (q_empty, count 2).
    if (lane == 0) {
      const int w = warp - (2 + 4 * NWG);  // 0: dV += P^T dO, 1: dK += dS^T Q
      constexpr uint32_t IDESC_G = idesc_bf16(KBM, D, true);
      const uint64_t qt_desc_mn = sdesc_sw128(sbase + C::OFF_Q, KBN * 128, 1024);   // MN-major Q/dO tiles
      const uint32_t d_tm = tmem + (w == 0 ? C::TM_DV : C::TM_DK);
      const uint32_t a_tm = tmem + (w == 0 ? C::TM_S : C::TM_DP);
      const uint32_t b_off = w == 0 ? C::QT_BYTES : 0;  // dO (for dV) or Q (for dK)
      bool ok = true;
      for (int i = 0; ok && i < n_q; ++i) {
        const int st = i % C::NSTAGE, bf = i % NBUF;
        ok = mbar_wait(&p_full[bf], (i / NBUF) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t b_desc = sdesc_add(qt_desc_mn, st * C::STAGE_BYTES + b_off);
#pragma unroll
        for (int kk = 0; kk < KBN / 16; ++kk)
          mma_bf16_ts(d_tm, a_tm + bf * KBN + packed_col<NWG>(kk), sdesc_add(b_desc, kk * 16 * 128), IDESC_G,
                      (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&q_empty[st]);
      }
      if (ok) mma_commit(last_done);
      if (!ok) {
        raise_abort(abort_flag, p.status);
        mma_commit(&drain_g[w]);
        volatile int never = 0;
        mbar_wait(&drain_g[w], 0, &never);
      }
    }
  } else {
    // ---------------------------------------------------------------- gradients (thread = key)
    const int wg = (warp - 2) >> 2;
    constexpr int NCOL = KBN / NWG;  // query columns of a tile this warpgroup forms
    const int kr = ((warp & 3) << 5) + lane;
    const int key = kb + kr;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      const int bf = i % NBUF;
      ok = warp_wait(&s_full[bf], (i / NBUF) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      const int st = i % C::NSTAGE;
      const float4* sl = stat + st * (KBN / 2);
      const int p0 = (qt0 + i) * Pq;
      const bool diag = p0 + p.delta < kb + KBM;  // some rows of this tile precede some keys
      // P^T of this warpgroup's columns from S^T first, while dP^T may still be computed
      float e[NCOL];
#pragma unroll
      for (int hf = 0; hf < NCOL / 32; ++hf) {
        const int c0 = wg * NCOL + hf * 32;
        uint32_t s[32];
        tmem_ld32(tmem + lane_base + C::TM_S + bf * KBN + c0, s);
        float* ee = e + hf * 32;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float4 rs = sl[(c0 + c) >> 1];  // rows c0+c, c0+c+1: {-lse2, Delta, -lse2, Delta}
          ffma2(__uint_as_float(s[c]), __uint_as_float(s[c + 1]), sl2, sl2, rs.x, rs.z, ee[c], ee[c + 1]);
          ee[c] = ex2(ee[c]);
          ee[c + 1] = ex2(ee[c + 1]);
        }
        if (diag) {
          // row r sits at position p0 + r % Pq (head-major tile); keys after it (+ delta) are masked
          const int dk = key - p.delta - p0;
          if ((Pq & (Pq - 1)) == 0) {
#pragma unroll
            for (int c = 0; c < 32; ++c) ee[c] = (dk > ((c0 + c) & (Pq - 1))) ? 0.f : ee[c];
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) ee[c] = (dk > (c0 + c) % Pq) ? 0.f : ee[c];
          }
        }
      }
      ok = warp_wait(&dp_full[bf], (i / NBUF) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      uint32_t pp[NCOL / 2], pd[NCOL / 2];
#pragma unroll
      for (int hf = 0; hf < NCOL / 32; ++hf) {
        const int c0 = wg * NCOL + hf * 32;
        uint32_t dpv[32];
        tmem_ld32(tmem + lane_base + C::TM_DP + bf * KBN + c0, dpv);
        const float* ee = e + hf * 32;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float4 rs = sl[(c0 + c) >> 1];
          float d0, d1;
          fsubmul2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1]), rs.y, rs.w, ee[c], ee[c + 1], d0, d1);
          pp[hf * 16 + (c >> 1)] = pack_bf16(ee[c], ee[c + 1]);
          pd[hf * 16 + (c >> 1)] = pack_bf16(d0, d1);
        }
      }
      if constexpr (NCOL == 64) {
        tmem_st32x2(tmem + lane_base + C::TM_S + bf * KBN, tmem + lane_base + C::TM_DP + bf * KBN, pp, pd);
      } else {
        // over this warpgroup's own S^T / dP^T columns (see packed_col)
        tmem_st16(tmem + lane_base + C::TM_S + bf * KBN + wg * 32, pp);
        tmem_st16(tmem + lane_base + C::TM_DP + bf * KBN + wg * 32, pd);
      }
      tc_fence_before();
      mbar_arrive(&p_full[bf]);
    }
    if (!ok) {
      raise_abort(abort_flag, p.status);
    } else {
      ok = warp_wait(last_done, 0, abort_flag);
      if (!ok) {
        raise_abort(abort_flag, p.status);
      } else {
        tc_fence_after();
        // dV (WG 0 / first half) and dK (scaled; WG 1 / second half)
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {
          if (NWG == 2 && part != wg) continue;
          const uint32_t src = part == 0 ? C::TM_DV : C::TM_DK;
          const int64_t orow = (static_cast<int64_t>(bg) * p.Tk + (key < p.Tk ? key : 0)) * D;
          __nv_bfloat16* out = (part == 0 ? p.dv : p.dk) + orow;
          float* out_acc = p.dk_acc != nullptr ? (part == 0 ? p.dv_acc : p.dk_acc) + orow : nullptr;
          const float mul = part == 0 ? 1.f : p.scale;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t acc[32];
            tmem_ld32(tmem + lane_base + src + c0, acc);
            if (key < p.Tk && out_acc != nullptr) {
              float4* dst = reinterpret_cast<float4*>(out_acc + c0);
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                float4 y = dst[u];
                y.x = fmaf(__uint_as_float(acc[4 * u]), mul, y.x);
                y.y = fmaf(__uint_as_float(acc[4 * u + 1]), mul, y.y);
                y.z = fmaf(__uint_as_float(acc[4 * u + 2]), mul, y.z);
                y.w = fmaf(__uint_as_float(acc[4 * u + 3]), mul, y.w);
                dst[u] = y;
              }
            } else if (key < p.Tk) {
              uint4* dst = reinterpret_cast<uint4*>(out + c0);
#pragma unroll
              for (int u = 0; u < 4; ++u)
                dst[u] = make_uint4(
                    pack_bf16(__uint_as_float(acc[8 * u]) * mul, __uint_as_float(acc[8 * u + 1]) * mul),
                    pack_bf16(__uint_as_float(acc[8 * u + 2]) * mul, __uint_as_float(acc[8 * u + 3]) * mul),
                    pack_bf16(__uint_as_float(acc[8 * u + 4]) * mul, __uint_as_float(acc[8 * u + 5]) * mul),
                    pack_bf16(__uint_as_float(acc[8 * u + 6]) * mul, __uint_as_float(acc[8 * u + 7]) * mul));
            }
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ============================================================================ dK / dV, d = 64
// CTA: 128 keys [kb, kb+128) of (b, g).  Query tiles of 128 rows, head-major inside the
// tile (row r -> head g*G + r/P2, position p0 + r%P2, P2 = floor(128/G)), so the S^T and
// dP^T products have N = 128.  One CTA per SM, 352 threads.
// TMEM (512 columns): S^T [0,128), dP^T [128,256), P^T [256,320) and dS^T [320,384)
// (bf16 pairs), dV [384,448), dK [448,512).  The gradient warps release S^T/dP^T as soon
// as they have read them (s_free), so S^T and dP^T of tile i+1 are computed while P^T and
// dS^T of tile i are formed; dV, dK of tile i follow (p_full), and their commit (q_empty)
// frees both the Q/dO stage and P^T, dS^T.
// Warps: 0 loads, 1 issues S^T and dP^T, 10 issues dV, 11 issues dK, 2..9 gradient warps:
// warpgroup w forms query columns [64w, 64w+64) of every tile; thread = key = TMEM lane.
// Three issuing threads: one waiting on a barrier (Q/dO loads and S^T released; P^T, dS^T
// written) does not leave the tensor pipe's short queue empty, and the N = 64 gradient
// products, which one thread issues more slowly than the pipe executes them, come from two.
constexpr int K2N = 128;

struct Dkv64Cfg {
  static constexpr int D = 64;
  static constexpr int THREADS = 64 + 256 + 64;
  static constexpr int KV_BYTES = KBM * D * 2;    // the CTA's K (or V) tile
  static constexpr int QT_BYTES = K2N * D * 2;    // one 128-row Q (or dO) tile
  static constexpr int NSTAGE = 4;
  static constexpr int STAGE_BYTES = 2 * QT_BYTES;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_BYTES;
  static constexpr int OFF_Q = 2 * KV_BYTES;      // stage s: Q at + s*STAGE, dO at + QT_BYTES
  static constexpr int OFF_STAT = OFF_Q + NSTAGE * STAGE_BYTES;  // [NSTAGE][128] {-lse*log2e, Delta}
  static constexpr int OFF_BAR = OFF_STAT + NSTAGE * K2N * 8;
  // kv_full, q_full[NSTAGE], q_empty[NSTAGE], s_full, s_free, p_full, drain_g[2], drain, last_done
  static constexpr int NBAR = 1 + 2 * NSTAGE + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_P = 256, TM_DS = 320, TM_DV = 384, TM_DK = 448;
  static constexpr uint32_t TM_COLS = 512;
};

__global__ void __launch_bounds__(Dkv64Cfg::THREADS, 1)
    moda_bwd_dkdv64_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                           const BwdTcParams p) {
  using C = Dkv64Cfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P2 = K2N / p.G;  // positions per query tile
  const int ngroups = p.B * p.Hkv;
  int kblk, bg;
  kv_block_of(static_cast<int>(blockIdx.x), ngroups, (p.Tk + KBM - 1) / KBM, kblk, bg);
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int kb = kblk * KBM;
  const int qt0 = max(kb - p.delta, 0) / P2, qt1 = (p.T - 1) / P2;
  const int n_q = qt1 - qt0 + 1;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + C::NSTAGE;
  uint64_t* s_full = q_empty + C::NSTAGE;
  uint64_t* s_free = s_full + 1;
  uint64_t* p_full = s_free + 1;
  uint64_t* drain_g = p_full + 1;  // [2]: one per gradient-product issuer
  uint64_t* drain = p_full + 3;
  uint64_t* last_done = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  // per stage: -lse*log2(e) of the 128 rows, then Delta of the 128 rows (four rows per float4)
  const float4* stat = reinterpret_cast<const float4*>(smem + C::OFF_STAT);

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(&q_full[i], 1 + 32);  // TMA arrive + one cp.async arrival per producer lane
      mbar_init(&q_empty[i], 2);      // the dV and the dK issuer
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 8);  // one arrival per gradient warp
    mbar_init(p_full, 8);
    mbar_init(drain, 1);
    mbar_init(&drain_g[0], 1);
    mbar_init(&drain_g[1], 1);
    mbar_init(last_done, 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // rows past P2*G of every query tile are never written by TMA: zero them once
  if (P2 * p.G < K2N) {
    for (int i = threadIdx.x; i < C::NSTAGE * C::STAGE_BYTES / 16; i += blockDim.x)
      st_shared_v4(sbase + C::OFF_Q + i * 16, make_uint4(0, 0, 0, 0));
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmO);
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
    // ---------------------------------------------------------------- loads
    bool ok = true;
    int issued = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
      tma_load_3d(smem + C::OFF_K, &tmK, kv_full, 0, kb, bg);
      tma_load_3d(smem + C::OFF_V, &tmV, kv_full, 0, kb, bg);
    }
    for (int i = 0; i < n_q; ++i) {
      const int st = i % C::NSTAGE, use = i / C::NSTAGE;
      if (use > 0 && !warp_wait(&q_empty[st], (use - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const int p0 = (qt0 + i) * P2;
      // row statistics (LSE, Delta) of this tile, copied asynchronously.  Rows that do not
      // exist (head >= G or position >= T) read a valid row's statistics: their Q and dO rows
      // are zero in shared memory, so whatever finite P and dS they get contributes nothing.
      const uint32_t sl = sbase + C::OFF_STAT + st * K2N * 8;
#pragma unroll
      for (int rr = 0; rr < K2N / 32; ++rr) {
        const int r = lane + 32 * rr;
        const int hh = min(r / P2, p.G - 1), pos = min(p0 + r % P2, p.T - 1);
        const int64_t row = (static_cast<int64_t>(b) * p.H + g * p.G + hh) * p.T + pos;
        const float* src = reinterpret_cast<const float*>(p.stats + row);
        cp_async_4(sl + r * 4, src);
        cp_async_4(sl + K2N * 4 + r * 4, src + 1);
      }
      cp_async_arrive_noinc(&q_full[st]);
      if (lane == 0) {
        uint8_t* dst = smem + C::OFF_Q + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&q_full[st], static_cast<uint32_t>(2 * P2 * p.G * D * 2));
        tma_load_3d(dst, &tmQ, &q_full[st], 0, p0, b * p.H + g * p.G);
        tma_load_3d(dst + C::QT_BYTES, &tmO, &q_full[st], 0, p0, b * p.H + g * p.G);
      }
      issued = i + 1;
    }
    if (!ok || *abort_flag) {
      if (lane == 0) {
        raise_abort(abort_flag, p.status);
        volatile int never = 0;
        mbar_wait(kv_full, 0, &never);
      }
      volatile int never = 0;
      for (int i = max(0, issued - C::NSTAGE); i < issued; ++i)
        mbar_wait(&q_full[i % C::NSTAGE], (i / C::NSTAGE) & 1, &never);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- S^T, dP^T issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(KBM, K2N, false);
      const uint64_t k_desc = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
      const uint64_t qt_desc_k = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);  // K-major Q/dO tiles
      bool ok = mbar_wait(kv_full, 0, abort_flag);
      for (int i = 0; ok && i < n_q; ++i) {
        // S^T(i) = K Q_i^T and dP^T(i) = V dO_i^T, once tile i is loaded and the gradient
        // warps have read S^T/dP^T of tile i-1
        const int st = i % C::NSTAGE;
        ok = mbar_wait(&q_full[st], (i / C::NSTAGE) & 1, abort_flag) &&
             (i == 0 || mbar_wait(s_free, (i - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint64_t q_desc = sdesc_add(qt_desc_k, st * C::STAGE_BYTES);
        const uint64_t o_desc = sdesc_add(q_desc, C::QT_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tmem + C::TM_S, sdesc_add(k_desc, kk * 32), sdesc_add(q_desc, kk * 32), IDESC_S, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tmem + C::TM_DP, sdesc_add(v_desc, kk * 32), sdesc_add(o_desc, kk * 32), IDESC_S, kk > 0);
        mma_commit(s_full);
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
      }
    }
  } else if (warp == 10 || warp == 11) {
    // ---------------------------------------------------------------- dV (warp 10), dK (warp 11) issuers
    // dV, dK of tile j follow p_full(j), which the gradient warps signal only after reading
    // S^T(j), dP^T(j): those MMAs have completed, so each thread's commit after its product
    // of tile j is its last use of the Q/dO stage and of P^T (dS^T); q_empty completes when
    // both have committed.
    if (lane == 0) {
      const int w = warp - 10;  // 0: dV += P^T dO, 1: dK += dS^T Q
      constexpr uint32_t IDESC_G = idesc_bf16(KBM, D, true);
      const uint64_t qt_desc_mn = sdesc_sw128(sbase + C::OFF_Q, K2N * 128, 1024);  // MN-major Q/dO tiles
      const uint32_t d_tm = tmem + (w == 0 ? C::TM_DV : C::TM_DK);
      const uint32_t a_tm = tmem + (w == 0 ? C::TM_P : C::TM_DS);
      const uint32_t b_off = w == 0 ? C::QT_BYTES : 0;  // dO (for dV) or Q (for dK)
      bool ok = true;
      for (int j = 0; ok && j < n_q; ++j) {
        const int st = j % C::NSTAGE;
        ok = mbar_wait(p_full, j & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t b_desc = sdesc_add(qt_desc_mn, st * C::STAGE_BYTES + b_off);
#pragma unroll
        for (int kk = 0; kk < K2N / 16; ++kk)
          mma_bf16_ts(d_tm, a_tm + kk * 8, sdesc_add(b_desc, kk * 16 * 128), IDESC_G, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&q_empty[st]);  // also tells the gradient warps that P^T(j) (dS^T(j)) is read
      }
      if (ok) mma_commit(last_done);
      if (!ok) {
        raise_abort(abort_flag, p.status);
        mma_commit(&drain_g[w]);
        volatile int never = 0;
        mbar_wait(&drain_g[w], 0, &never);
      }
    }
  } else {
    // ---------------------------------------------------------------- gradients (thread = key)
    const int wg = (warp - 2) >> 2;
    const int kr = ((warp & 3) << 5) + lane;
    const int key = kb + kr;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool pow2 = (P2 & (P2 - 1)) == 0;
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      ok = warp_wait(s_full, i & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      uint32_t s[64], dpv[64];
      tmem_ld64x2(tmem + lane_base + C::TM_S + wg * 64, tmem + lane_base + C::TM_DP + wg * 64, s, dpv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      const int st = i % C::NSTAGE;
      const float4* sl = stat + st * (K2N / 2);  // [0, 32): -lse2 of rows 4c..4c+3; [32, 64): Delta
      const int p0 = (qt0 + i) * P2;
      const bool diag = p0 + p.delta < kb + KBM;  // some rows of this tile precede some keys
      const int dk = key - p.delta - p0;
      // P^T and dS^T of both 32-column halves first, in registers; only then wait until the
      // dV/dK products of tile i-1 have read the single P^T, dS^T buffer (their commit
      // completes tile i-1's phase of q_empty), so that wait overlaps this tile's arithmetic
      uint32_t pp[32], pd[32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int c0 = wg * 64 + hf * 32;  // first query column of this group
        float e[32];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 ls = sl[(c0 + c) >> 2];  // -lse2 of rows c0+c .. c0+c+3
          ffma2(__uint_as_float(s[hf * 32 + c]), __uint_as_float(s[hf * 32 + c + 1]), sl2, sl2, ls.x, ls.y, e[c],
                e[c + 1]);
          ffma2(__uint_as_float(s[hf * 32 + c + 2]), __uint_as_float(s[hf * 32 + c + 3]), sl2, sl2, ls.z, ls.w,
                e[c + 2], e[c + 3]);
#pragma unroll
          for (int u = 0; u < 4; ++u) e[c + u] = ex2(e[c + u]);
        }
        if (diag) {
          // row r sits at position p0 + r % P2 (head-major tile); keys after it are masked
          if (pow2) {
#pragma unroll
            for (int c = 0; c < 32; ++c) e[c] = (dk > ((c0 + c) & (P2 - 1))) ? 0.f : e[c];
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) e[c] = (dk > (c0 + c) % P2) ? 0.f : e[c];
          }
        }
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 dl = sl[K2N / 4 + ((c0 + c) >> 2)];  // Delta of rows c0+c .. c0+c+3
          float d0, d1, d2, d3;
          fsubmul2(__uint_as_float(dpv[hf * 32 + c]), __uint_as_float(dpv[hf * 32 + c + 1]), dl.x, dl.y, e[c],
                   e[c + 1], d0, d1);
          fsubmul2(__uint_as_float(dpv[hf * 32 + c + 2]), __uint_as_float(dpv[hf * 32 + c + 3]), dl.z, dl.w,
                   e[c + 2], e[c + 3], d2, d3);
          pp[hf * 16 + (c >> 1)] = pack_bf16(e[c], e[c + 1]);
          pp[hf * 16 + (c >> 1) + 1] = pack_bf16(e[c + 2], e[c + 3]);
          pd[hf * 16 + (c >> 1)] = pack_bf16(d0, d1);
          pd[hf * 16 + (c >> 1) + 1] = pack_bf16(d2, d3);
        }
      }
      if (i > 0) {
        ok = warp_wait(&q_empty[(i - 1) % C::NSTAGE], ((i - 1) / C::NSTAGE) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st32_nowait(tmem + lane_base + C::TM_P + wg * 32, pp);
      tmem_st32_nowait(tmem + lane_base + C::TM_DS + wg * 32, pd);
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (!ok) {
      raise_abort(abort_flag, p.status);
    } else {
      ok = warp_wait(last_done, 0, abort_flag);
      if (!ok) {
        raise_abort(abort_flag, p.status);
      } else {
        tc_fence_after();
        // dV (warpgroup 0) and dK (scaled; warpgroup 1)
        const uint32_t src = wg == 0 ? C::TM_DV : C::TM_DK;
        const int64_t orow = (static_cast<int64_t>(bg) * p.Tk + (key < p.Tk ? key : 0)) * D;
        __nv_bfloat16* out = (wg == 0 ? p.dv : p.dk) + orow;
        float* out_acc = p.dk_acc != nullptr ? (wg == 0 ? p.dv_acc : p.dk_acc) + orow : nullptr;
        const float mul = wg == 0 ? 1.f : p.scale;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t acc[32];
          tmem_ld32(tmem + lane_base + src + c0, acc);
          if (key < p.Tk && out_acc != nullptr) {
            float4* dst = reinterpret_cast<float4*>(out_acc + c0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float4 y = dst[u];
              y.x = fmaf(__uint_as_float(acc[4 * u]), mul, y.x);
              y.y = fmaf(__uint_as_float(acc[4 * u + 1]), mul, y.y);
              y.z = fmaf(__uint_as_float(acc[4 * u + 2]), mul, y.z);
              y.w = fmaf(__uint_as_float(acc[4 * u + 3]), mul, y.w);
              dst[u] = y;
            }
          } else if (key < p.Tk) {
            uint4* dst = reinterpret_cast<uint4*>(out + c0);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[u] = make_uint4(
                  pack_bf16(__uint_as_float(acc[8 * u]) * mul, __uint_as_float(acc[8 * u + 1]) * mul),
                  pack_bf16(__uint_as_float(acc[8 * u + 2]) * mul, __uint_as_float(acc[8 * u + 3]) * mul),
                  pack_bf16(__uint_as_float(acc[8 * u + 4]) * mul, __uint_as_float(acc[8 * u + 5]) * mul),
                  pack_bf16(__uint_as_float(acc[8 * u + 6]) * mul, __uint_as_float(acc[8 * u + 7]) * mul));
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ============================================================================ dQ, d = 64
// CTA: 128 expanded rows of (b, g), position-major (row r -> position p0 + r/G, head
// g*G + r%G), P = floor(128/G) positions.  Key tiles of 128, so S and dP have N = 128.
// One CTA per SM, 352 threads.  TMEM (512 columns): S [0,128), dP [128,256) (each
// completed and released through barriers of its own: P is formed from S while dP is
// still computed, and S and dP of tile j+1 are computed while dS of tile j is formed), dS[2] [256,320), [320,384) (bf16 pairs, double-buffered),
// dQ [384,448), Q [448,480) and dO [480,512) (bf16 pairs: the A operands of S and dP, so
// those products read only K and V from shared memory).  Warps: 0 loads K_j, V_j; 1
// issues S and dP; 10 issues dQ; 2..9 gradient warps (warpgroup w forms key columns
// [64w, 64w+64) of every tile; warpgroup 0 also writes Q and dO into TMEM).  Two issuing threads, because a thread that waits on a barrier lets
// the tensor pipe's short queue run dry: the S/dP thread waits for K/V and for the
// gradient warps to release S, the dQ thread for dS, each while the other's MMAs run.
constexpr int Q2N = 128;

struct Dq64Cfg {
  static constexpr int D = 64;
  static constexpr int THREADS = 64 + 256 + 32;
  static constexpr int KV_BYTES = Q2N * D * 2;  // one K (or V) tile; a ring slot holds both
  static constexpr int NSLOT = 3;
  static constexpr int OFF_KV = 0;
  // Q and dO of a block staged by TMA (128-byte swizzle) on their way into TMEM
  static constexpr int QS_BYTES = QBM * D * 2;
  static constexpr int OFF_QS = OFF_KV + NSLOT * 2 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_QS + 2 * QS_BYTES;
  // kv_full[NSLOT], kv_empty[NSLOT], q_full, s_full, s_free, ds_full, drain_dq, qs_full, drain, last_done,
  // dp_full, dp_free, qs_empty
  static constexpr int NBAR = 2 * NSLOT + 11;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16;
  // Q and dO of the CTA's rows stay in TMEM (A operands of S and dP, bf16 pairs)
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DS = 256, TM_DQ = 384, TM_Q = 448, TM_DO = 480;
  static constexpr uint32_t TM_COLS = 512;
};

__global__ void __launch_bounds__(Dq64Cfg::THREADS, 1)
    moda_bwd_dq64_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO,
                         const BwdTcParams p) {
  using C = Dq64Cfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) record_status(p.status, kStatusConfig);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = QBM / p.G;
  const int cta = static_cast<int>(blockIdx.x);
  const int n_blk = dq_blocks_of_cta((p.T + P - 1) / P * p.B * p.Hkv, p.n_cta, cta);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::NSLOT;
  uint64_t* q_full = bars + 2 * C::NSLOT;
  uint64_t* s_full = q_full + 1;
  uint64_t* s_free = s_full + 1;
  uint64_t* ds_full = s_free + 1;
  uint64_t* drain_dq = ds_full + 1;
  uint64_t* drain = ds_full + 3;
  uint64_t* last_done = drain + 1;
  uint64_t* dp_full = last_done + 1;  // S and dP complete, and are released, separately
  uint64_t* dp_free = dp_full + 1;
  uint64_t* qs_full = ds_full + 2;   // a block's Q and dO staged in shared memory
  uint64_t* qs_empty = dp_free + 1;  // ... and copied from there into TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(qs_full, 1);
    mbar_init(qs_empty, 128);  // warpgroup 0 of the gradient warps
    mbar_init(q_full, 128);
    mbar_init(s_full, 1);
    mbar_init(s_free, 8);  // one arrival per gradient warp
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 8);
    mbar_init(ds_full, 8);
    mbar_init(drain, 1);
    mbar_init(drain_dq, 1);
    mbar_init(last_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Barrier phases and ring slots follow the running count of key tiles over the CTA's
  // blocks (it), q_full and last_done the block count (k).
  if (warp == 0) {
    // ---------------------------------------------------------------- K_j, V_j loads
    // (the loads of the next block start while this block's last tiles are processed)
    if (lane == 0) {
      int it = 0, staged = 0;
      bool ok = true;
      for (int k = 0; ok && k < n_blk; ++k) {
        const DqBlock x = dq_block_at(p, P, cta, k, Q2N);
        // this block's Q and dO rows (position-major, positions past T read as zeros) into
        // the staging buffer, once the previous block's have been copied out of it
        if (k > 0 && !mbar_wait(qs_empty, (k - 1) & 1, abort_flag)) {
          raise_abort(abort_flag, p.status);
          break;
        }
        mbar_arrive_expect_tx(qs_full, 2u * p.G * P * 128u);
        tma_load_4d(smem + C::OFF_QS, &tmQ, qs_full, 0, x.g * p.G, x.p0, x.b);
        tma_load_4d(smem + C::OFF_QS + C::QS_BYTES, &tmO, qs_full, 0, x.g * p.G, x.p0, x.b);
        staged = k + 1;
        for (int j = 0; j < x.n_kv; ++j, ++it) {
          const int slot = it % C::NSLOT, use = it / C::NSLOT;
          if (use > 0 && !mbar_wait(&kv_empty[slot], (use - 1) & 1, abort_flag)) {
            raise_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          uint8_t* dst = smem + C::OFF_KV + slot * 2 * C::KV_BYTES;
          mbar_arrive_expect_tx(&kv_full[slot], 2 * C::KV_BYTES);
          tma_load_3d(dst, &tmK, &kv_full[slot], 0, j * Q2N, x.bg);
          tma_load_3d(dst + C::KV_BYTES, &tmV, &kv_full[slot], 0, j * Q2N, x.bg);
        }
      }
      if (*abort_flag) {
        volatile int never = 0;
        for (int j = max(0, it - C::NSLOT); j < it; ++j) mbar_wait(&kv_full[j % C::NSLOT], (j / C::NSLOT) & 1, &never);
        if (staged > 0) mbar_wait(qs_full, (staged - 1) & 1, &never);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- S, dP issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_bf16(QBM, Q2N, false);
      const uint64_t kv_desc_k = sdesc_sw128(sbase + C::OFF_KV, 16, 1024);  // K-major
      bool ok = true;
      int it = 0;
      for (int k = 0; ok && k < n_blk; ++k) {
        const int n_kv = dq_block_at(p, P, cta, k, Q2N).n_kv;
        ok = mbar_wait(q_full, k & 1, abort_flag);  // Q and dO of this block in TMEM
        for (int j = 0; ok && j < n_kv; ++j, ++it) {
          // S = Q K_j^T once K_j, V_j are loaded and the gradient warps have read the
          // previous S; dP = dO V_j^T once they have read the previous dP
          const int slot = it % C::NSLOT;
          ok = mbar_wait(&kv_full[slot], (it / C::NSLOT) & 1, abort_flag) &&
               (it == 0 || mbar_wait(s_free, (it - 1) & 1, abort_flag));
          if (!ok) break;
          tc_fence_after();
          const uint64_t k_desc = sdesc_add(kv_desc_k, slot * 2 * C::KV_BYTES);
          const uint64_t v_desc = sdesc_add(k_desc, C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ts(tmem + C::TM_S, tmem + C::TM_Q + kk * 8, sdesc_add(k_desc, kk * 32), IDESC_S, kk > 0);
          mma_commit(s_full);
          ok = it == 0 || mbar_wait(dp_free, (it - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_bf16_ts(tmem + C::TM_DP, tmem + C::TM_DO + kk * 8, sdesc_add(v_desc, kk * 32), IDESC_S, kk > 0);
          mma_commit(dp_full);
        }
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
      }
    }
  } else if (warp == 10) {
    // ---------------------------------------------------------------- dQ issuer
    // dQ(j) is issued after ds_full(j), which the gradient warps signal only after reading
    // S(j), dP(j): those MMAs have completed, so this thread's commit after dQ(j) is the
    // last use of K_j, V_j and frees their slot.  The first dQ of a block overwrites the
    // accumulator: the gradient warps signal its ds_full only after their epilogue of the
    // previous block has read it.
    if (lane == 0) {
      constexpr uint32_t IDESC_DQ = idesc_bf16(QBM, D, true);
      const uint64_t kv_desc_mn = sdesc_sw128(sbase + C::OFF_KV, Q2N * 128, 1024);  // MN-major
      bool ok = true;
      int it = 0;
      for (int k = 0; ok && k < n_blk; ++k) {
        const int n_kv = dq_block_at(p, P, cta, k, Q2N).n_kv;
        for (int j = 0; j < n_kv; ++j, ++it) {
          const int slot = it % C::NSLOT;
          ok = mbar_wait(ds_full, it & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t k_desc = sdesc_add(kv_desc_mn, slot * 2 * C::KV_BYTES);
          const uint32_t ds = C::TM_DS + (it & 1) * 64;
#pragma unroll
          for (int kk = 0; kk < Q2N / 16; ++kk)
            mma_bf16_ts(tmem + C::TM_DQ, tmem + ds + kk * 8, sdesc_add(k_desc, kk * 16 * 128), IDESC_DQ,
                        (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&kv_empty[slot]);  // K_j, V_j and dS(j) no longer read
        }
        if (ok) mma_commit(last_done);  // this block's dQ is complete
      }
      if (!ok) {
        raise_abort(abort_flag, p.status);
        mma_commit(drain_dq);
        volatile int never = 0;
        mbar_wait(drain_dq, 0, &never);
      }
    }
  } else {
    // ---------------------------------------------------------------- gradients (thread = row)
    const int wg = (warp - 2) >> 2;
    const int r = ((warp & 3) << 5) + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool row_in = r < P * p.G;
    const float sl2 = p.scale_log2;
    // row r of Q and dO of block k into TMEM lane r (the A operands of S and dP): column c
    // holds elements 2c, 2c+1, i.e. the row's 32-bit words as stored.  The rows come from
    // the staging buffer (row r: 128 bytes, 16-byte chunk c at chunk c ^ (r % 8)); rows past
    // P*G, which the TMA box does not cover, are zero.
    auto load_q = [&](int k) -> bool {
      if (!warp_wait(qs_full, k & 1, abort_flag)) return false;
      const uint32_t qs = sbase + C::OFF_QS + r * 128;
      uint32_t qw[32], ow[32];
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {
        const uint32_t off = static_cast<uint32_t>((ch ^ (r & 7)) << 4);
        const uint4 a = row_in ? ld_shared_v4(qs + off) : make_uint4(0, 0, 0, 0);
        const uint4 o = row_in ? ld_shared_v4(qs + C::QS_BYTES + off) : make_uint4(0, 0, 0, 0);
        qw[4 * ch] = a.x;
        qw[4 * ch + 1] = a.y;
        qw[4 * ch + 2] = a.z;
        qw[4 * ch + 3] = a.w;
        ow[4 * ch] = o.x;
        ow[4 * ch + 1] = o.y;
        ow[4 * ch + 2] = o.z;
        ow[4 * ch + 3] = o.w;
      }
      mbar_arrive(qs_empty);
      tmem_st32_nowait(tmem + lane_base + C::TM_Q, qw);
      tmem_st32_nowait(tmem + lane_base + C::TM_DO, ow);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_full);
      return true;
    };
    // global row of thread r in block k, and whether it exists
    auto row_of = [&](int k, bool& valid) -> int64_t {
      const DqBlock x = dq_block_at(p, P, cta, k, Q2N);
      const int pos = x.p0 + r / p.G;
      valid = row_in && pos < p.T;
      return (static_cast<int64_t>(x.b) * p.H + x.g * p.G + r % p.G) * p.T + (valid ? pos : 0);
    };
    bool ok = !(wg == 0 && n_blk > 0) || load_q(0);
    int it = 0;
    // row statistics of the next block, loaded while this block runs
    float2 stt_next = make_float2(-INFINITY, 0.f);
    if (n_blk > 0) {
      bool v0;
      const int64_t r0 = row_of(0, v0);
      if (v0) stt_next = p.stats[r0];
    }
    for (int k = 0; ok && k < n_blk; ++k) {
      const DqBlock x = dq_block_at(p, P, cta, k, Q2N);
      const int pos = x.p0 + r / p.G;
      const bool valid = row_in && pos < p.T;
      const int h = x.g * p.G + r % p.G;
      const int64_t row = (static_cast<int64_t>(x.b) * p.H + h) * p.T + (valid ? pos : 0);
      const float2 stt = stt_next;
      // the depth share this thread adds in the epilogue (one 128-byte line) into L2 now
      if (p.S > 0 && valid) prefetch_l2(p.dq_accum + row * D + wg * 32);
      const float nlse2 = stt.x;  // -lse * log2(e)
      const float dlt = stt.y;
      const int key_end = min(pos + p.delta, p.Tk - 1);  // last key this row sees
      for (int j = 0; j < x.n_kv; ++j, ++it) {
        ok = warp_wait(s_full, it & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        // the dS buffer (it & 1) is free once the dQ product two tiles earlier has read it (its
        // commit completes that tile's phase of kv_empty): tested now, waited for only if not
        const bool ds_free = it < 2 || mbar_test_wait(&kv_empty[(it - 2) % C::NSLOT], ((it - 2) / C::NSLOT) & 1);
        // P from S first, while dP may still be computed; then dS = P (dP - Delta)
        float e[64];
        {
          uint32_t s[64];
          tmem_ld64(tmem + lane_base + C::TM_S + wg * 64, s);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free);
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            ffma2(__uint_as_float(s[c]), __uint_as_float(s[c + 1]), sl2, sl2, nlse2, nlse2, e[c], e[c + 1]);
            e[c] = ex2(e[c]);
            e[c + 1] = ex2(e[c + 1]);
          }
          const int lim = valid ? key_end - (j * Q2N + wg * 64) : -1;  // columns c <= lim are visible
          if (lim < 63) {
#pragma unroll
            for (int c = 0; c < 64; ++c) e[c] = (c <= lim) ? e[c] : 0.f;
          }
        }
        ok = warp_wait(dp_full, it & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        uint32_t dpv[64];
        tmem_ld64(tmem + lane_base + C::TM_DP + wg * 64, dpv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dp_free);
        const uint32_t ds = C::TM_DS + (it & 1) * 64 + wg * 32;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float d0, d1;
            fsubmul2(__uint_as_float(dpv[hf * 32 + c]), __uint_as_float(dpv[hf * 32 + c + 1]), dlt, dlt,
                     e[hf * 32 + c], e[hf * 32 + c + 1], d0, d1);
            pk[c >> 1] = pack_bf16(d0, d1);
          }
          if (hf == 0 && it >= 2) {
            if (!__all_sync(0xffffffffu, ds_free)) {
              ok = warp_wait(&kv_empty[(it - 2) % C::NSLOT], ((it - 2) / C::NSLOT) & 1, abort_flag);
              if (!ok) break;
            }
            tc_fence_after();
          }
          tmem_st16_nowait(tmem + lane_base + ds + hf * 16, pk);
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full);
      }
      if (!ok) break;
      // the S and dP products of this block have completed (their results were read): Q and
      // dO of the next block replace theirs first, so that the next block's products can
      // start while this block's epilogue runs
      if (wg == 0 && k + 1 < n_blk && !load_q(k + 1)) {
        ok = false;
        break;
      }
      // warpgroup w writes dq columns [32w, 32w+32); the depth share of those columns and the
      // next block's row statistics are loaded before the wait for the last dQ product
      const int c0 = wg * 32;
      float extra[32];
      if (p.S > 0 && valid) {
        const float4* src = reinterpret_cast<const float4*>(p.dq_accum + row * D + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 e4 = src[i];
          extra[4 * i] = e4.x;
          extra[4 * i + 1] = e4.y;
          extra[4 * i + 2] = e4.z;
          extra[4 * i + 3] = e4.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) extra[i] = 0.f;
      }
      if (k + 1 < n_blk) {
        bool vn;
        const int64_t rn = row_of(k + 1, vn);
        stt_next = vn ? p.stats[rn] : make_float2(-INFINITY, 0.f);
      }
      ok = warp_wait(last_done, k & 1, abort_flag);
      if (!ok) break;
      tc_fence_after();
      uint32_t acc[32];
      tmem_ld32(tmem + lane_base + C::TM_DQ + c0, acc);
      if (valid && p.dq_acc != nullptr) {
        float4* dst = reinterpret_cast<float4*>(p.dq_acc + row * D + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 y = dst[i];
          y.x += fmaf(__uint_as_float(acc[4 * i]), p.scale, extra[4 * i]);
          y.y += fmaf(__uint_as_float(acc[4 * i + 1]), p.scale, extra[4 * i + 1]);
          y.z += fmaf(__uint_as_float(acc[4 * i + 2]), p.scale, extra[4 * i + 2]);
          y.w += fmaf(__uint_as_float(acc[4 * i + 3]), p.scale, extra[4 * i + 3]);
          dst[i] = y;
        }
      } else if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.dq + row * D + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t w[4];
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            const int c = 8 * i + 2 * k2;
            w[k2] = pack_bf16(fmaf(__uint_as_float(acc[c]), p.scale, extra[c]),
                              fmaf(__uint_as_float(acc[c + 1]), p.scale, extra[c + 1]));
          }
          dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // the accumulator read is complete (tcgen05.ld waits) before this warp's next ds_full
      tc_fence_before();
    }
    if (!ok) raise_abort(abort_flag, p.status);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ============================================================================ host
int bwd_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
}

// bf16 [planes][T][D] as the 3-D tensor (D, T, planes), box 64 x rows x depth, 128-byte
// swizzle, out-of-range rows read as zeros.
bool make_map(CUtensorMap* map, const void* base, int D, int T, int planes, int rows, int depth) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), static_cast<cuuint32_t>(depth)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q (or dO) [B][H][T][D] bf16 described as (D, H, T, B) -- heads before positions -- so that a
// box 64 x G x P x 1 lands position-major (row = position * G + head); positions past T read
// as zeros.
bool make_qpos_map(CUtensorMap* map, const void* base, int D, int T, int H, int B, int P, int G) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(T) * D * 2, static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H) * T * D * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(P), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_all(const BwdArgs& a, cudaStream_t s) {
  const Problem& pr = a.p;
  BwdTcParams p;
  p.B = pr.B;
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.T = pr.T;
  p.Tk = pr.Tk;
  p.delta = pr.delta;
  p.S = pr.S;
  p.S_read = pr.S_read;
  p.G = pr.G;
  p.scale = pr.scale;
  p.scale_log2 = pr.scale_log2;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.kd = static_cast<const __nv_bfloat16*>(a.kd);
  p.vd = static_cast<const __nv_bfloat16*>(a.vd);
  p.dout = static_cast<const __nv_bfloat16*>(a.dout);
  p.lse = a.lse;
  p.stats = a.stats;
  p.o = static_cast<const __nv_bfloat16*>(a.o);
  p.dq_accum = a.dq_accum;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.dkd = static_cast<__nv_bfloat16*>(a.dkd);
  p.dvd = static_cast<__nv_bfloat16*>(a.dvd);
  p.dq_acc = a.dq_acc;
  p.dk_acc = a.dk_acc;
  p.dv_acc = a.dv_acc;
  p.status = a.status;

  // stage 0: Delta (its own kernel only when S = 0; otherwise the depth kernel forms the
  // row statistics); stage 1: depth gradients; stage 2: dK/dV; stage 3: dQ (needs stage
  // 1's depth share of dQ).
  cudaError_t e = cudaSuccess;
  mark_event(a, 0, s);
  if (pr.S == 0) {
    e = launch_bwd_delta(a, 1, s);
    if (e != cudaSuccess) return e;
  }
  mark_event(a, 1, s);
  const int64_t positions = static_cast<int64_t>(pr.B) * pr.Hkv * pr.T;
  mark_event(a, 2, s);
  if (pr.S > 0) {
    const unsigned grid = static_cast<unsigned>((positions + 7) / 8);
    if (pr.G == 1) moda_bwd_depth_kernel<D, 1><<<grid, 256, 0, s>>>(p);
    else if (pr.G == 2) moda_bwd_depth_kernel<D, 2><<<grid, 256, 0, s>>>(p);
    else if (pr.G <= 4) moda_bwd_depth_kernel<D, 4><<<grid, 256, 0, s>>>(p);
    else moda_bwd_depth_kernel<D, 8><<<grid, 256, 0, s>>>(p);
    count_launches(1);
  }
  mark_event(a, 3, s);
  CUtensorMap tk128, tv128, tk64, tv64, tq, to;
  const int planes_kv = pr.B * pr.Hkv, planes_q = pr.B * pr.H;
  const int pq = KBN / pr.G;
  if (!make_map(&tk128, a.k, D, pr.Tk, planes_kv, KBM, 1) || !make_map(&tv128, a.v, D, pr.Tk, planes_kv, KBM, 1) ||
      !make_map(&tk64, a.k, D, pr.Tk, planes_kv, QBN, 1) || !make_map(&tv64, a.v, D, pr.Tk, planes_kv, QBN, 1) ||
      !make_map(&tq, a.q, D, pr.T, planes_q, pq, pr.G) || !make_map(&to, a.dout, D, pr.T, planes_q, pq, pr.G))
    return cudaErrorInvalidValue;
  const unsigned grid_kv = static_cast<unsigned>((pr.Tk + KBM - 1) / KBM) * planes_kv;
  const int P = QBM / pr.G;
  const unsigned grid_q = static_cast<unsigned>((pr.T + P - 1) / P) * planes_kv;
  if constexpr (D == 64) {
    // 128-column query / key tiles, S/dP released early, one CTA per SM (512 TMEM columns)
    CUtensorMap tq2, to2;
    const int pq2 = K2N / pr.G;
    if (!make_map(&tq2, a.q, D, pr.T, planes_q, pq2, pr.G) || !make_map(&to2, a.dout, D, pr.T, planes_q, pq2, pr.G))
      return cudaErrorInvalidValue;
    static std::atomic<uint64_t> smem_dkdv{0}, smem_dq{0};
    e = ensure_dynamic_smem(moda_bwd_dkdv64_kernel, Dkv64Cfg::SMEM, smem_dkdv);
    if (e != cudaSuccess) return e;
    e = ensure_dynamic_smem(moda_bwd_dq64_kernel, Dq64Cfg::SMEM, smem_dq);
    if (e != cudaSuccess) return e;
    mark_event(a, 4, s);
    moda_bwd_dkdv64_kernel<<<grid_kv, Dkv64Cfg::THREADS, Dkv64Cfg::SMEM, s>>>(tk128, tv128, tq2, to2, p);
    mark_event(a, 5, s);
    mark_event(a, 6, s);
    const int sms = bwd_sm_count();
    if (sms <= 0) return cudaErrorNoDevice;
    p.n_cta = static_cast<int>(std::min<unsigned>(grid_q, static_cast<unsigned>(sms)));
    CUtensorMap tq4, to4;
    if (!make_qpos_map(&tq4, a.q, D, pr.T, pr.H, pr.B, P, pr.G) || !make_qpos_map(&to4, a.dout, D, pr.T, pr.H, pr.B, P, pr.G))
      return cudaErrorInvalidValue;
    moda_bwd_dq64_kernel<<<p.n_cta, Dq64Cfg::THREADS, Dq64Cfg::SMEM, s>>>(tk128, tv128, tq4, to4, p);
    mark_event(a, 7, s);
  } else {
    // d = 128: 64-column tiles, double-buffered TMEM, two gradient warpgroups splitting
    // each tile's columns, one CTA per SM.
    using KC = DkvCfg<D, 2, 2>;
    using QC = DqCfg<D, 2, 2>;
    static std::atomic<uint64_t> smem_dkdv{0}, smem_dq{0};
    e = ensure_dynamic_smem(moda_bwd_dkdv_kernel<D, 2, 2>, KC::SMEM, smem_dkdv);
    if (e != cudaSuccess) return e;
    e = ensure_dynamic_smem(moda_bwd_dq_kernel<D, 2, 2>, QC::SMEM, smem_dq);
    if (e != cudaSuccess) return e;
    mark_event(a, 4, s);
    moda_bwd_dkdv_kernel<D, 2, 2><<<grid_kv, KC::THREADS, KC::SMEM, s>>>(tk128, tv128, tq, to, p);
    mark_event(a, 5, s);
    mark_event(a, 6, s);
    const int sms = bwd_sm_count();
    if (sms <= 0) return cudaErrorNoDevice;
    p.n_cta = static_cast<int>(std::min<unsigned>(grid_q, static_cast<unsigned>(sms)));
    CUtensorMap tq4, to4;
    if (!make_qpos_map(&tq4, a.q, D, pr.T, pr.H, pr.B, P, pr.G) || !make_qpos_map(&to4, a.dout, D, pr.T, pr.H, pr.B, P, pr.G))
      return cudaErrorInvalidValue;
    moda_bwd_dq_kernel<D, 2, 2><<<p.n_cta, QC::THREADS, QC::SMEM, s>>>(tk64, tv64, tq4, to4, p);
    mark_event(a, 7, s);
  }
  count_launches(2);
  return cudaGetLastError();
}

}  // namespace

// bf16, d in {64, 128}, 1 <= G <= 8 (the depth kernel keeps a position's G heads in registers).
bool bwd_sm103_supported(const Problem& p) { return (p.d == 64 || p.d == 128) && p.G >= 1 && p.G <= 8; }

cudaError_t launch_bwd_sm103(const BwdArgs& a, cudaStream_t s) {
  return a.p.d == 64 ? launch_all<64>(a, s) : launch_all<128>(a, s);
}

}  // namespace moda

