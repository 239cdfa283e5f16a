// Mixture-of-Depths Attention (MoDA): float64 CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
// statement of what the GPU library computes.  Only the test-suite, the smoke
// check and the benchmark's CPU-baseline leg may load it.  It shares no code,
// header, table or helper with the CUDA library, and the CUDA library never
// calls it.
//
// What it computes (MoDA, "One denominator allocates probability across both
// memories" frame, teaching form of paper Sec. 2.2 / Algorithm 1):
//   for one query head h at position t, with kv head g = h / G  (G = H / Hkv),
//     a_j = q_t . k_j / sqrt(d)           for sequence keys j <= t
//     b_i = q_t . kd_{i,t} / sqrt(d)      for the depth slots i of position t
//     o_t = (sum_j e^{a_j} v_j + sum_i e^{b_i} vd_{i,t})
//           / (sum_j e^{a_j} + sum_i e^{b_i})
// One softmax over the union of both key sets; the "Backup: grouped indexing"
// frame (Algorithm 1 / Sec. 3.3) fixes causal visibility (position >= key) and
// same-position depth visibility.  The oracle evaluates that definition row by
// row: gather every visible score, subtract the row maximum (an exact identity,
// used only to keep exp() finite), sum, divide once.  LSE = max + ln(sum).
//
// The backward is the analytic gradient of the same expression (the pages give
// none), evaluated per row and per key column:
//   P_s = exp(s - LSE_t),  D_t = dO_t . o_t,  dP_s = dO_t . v_s,
//   dS_s = P_s (dP_s - D_t)
//   dq_t = scale sum_s dS_s k_s ;  dk_j = scale sum_{h in g, t>=j} dS_tj q_t
//   dv_j = sum_{h in g, t>=j} P_tj dO_t ;  dkd_{i,t} = scale sum_{h in g} dS q_t
//   dvd_{i,t} = sum_{h in g} P dO_t
//
// All arithmetic is float64 with std::exp / std::log.  Inputs are read in their
// stored type (bf16 widened exactly, fp32 widened exactly, or fp64).
// Parity status: pinned (see the tests named test_oracle_*).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#include <sched.h>

namespace {

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

struct Dims {
  int64_t B, H, Hkv, T, S, d;
  double scale;       // <= 0 means 1/sqrt(d)
  int64_t seq_window; // 0: full causal window j <= t; w > 0: t-w < j <= t
  int32_t dtype;      // storage type of every input
  int32_t nthreads;   // <= 0: all cores in the affinity mask
};

struct In {
  const void *q, *k, *v, *kd, *vd, *dout;
};

inline double ld(const void* p, int dt, int64_t i) {
  if (dt == ORC_F64) return static_cast<const double*>(p)[i];
  if (dt == ORC_F32) return static_cast<double>(static_cast<const float*>(p)[i]);
  uint32_t u = static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

int cores_available() {
  cpu_set_t set;
  if (sched_getaffinity(0, sizeof set, &set) == 0) {
    int n = CPU_COUNT(&set);
    if (n > 0) return n;
  }
  unsigned hc = std::thread::hardware_concurrency();
  return hc ? static_cast<int>(hc) : 1;
}

int threads_for(const Dims& D) { return D.nthreads > 0 ? D.nthreads : cores_available(); }

// Runs fn(i) for i in [0, n) on a small pool with dynamic chunking.
template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
  if (n <= 0) return;
  if (nthreads <= 1 || n == 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      int64_t i = next.fetch_add(1);
      if (i >= n) break;
      fn(i);
    }
  };
  int nt = static_cast<int>(std::min<int64_t>(nthreads, n));
  std::vector<std::thread> pool;
  pool.reserve(nt - 1);
  for (int w = 1; w < nt; ++w) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
}

double scale_of(const Dims& D) { return D.scale > 0 ? D.scale : 1.0 / std::sqrt(static_cast<double>(D.d)); }

int64_t first_key(const Dims& D, int64_t t) {
  if (D.seq_window > 0) return std::max<int64_t>(0, t - D.seq_window + 1);
  return 0;
}

// Offsets of the rows/slabs in the dense row-major layouts.
int64_t off_q(const Dims& D, int64_t b, int64_t h, int64_t t) { return ((b * D.H + h) * D.T + t) * D.d; }
int64_t off_kv(const Dims& D, int64_t b, int64_t g, int64_t j) { return ((b * D.Hkv + g) * D.T + j) * D.d; }
int64_t off_dkv(const Dims& D, int64_t b, int64_t g, int64_t t, int64_t i) {
  return (((b * D.Hkv + g) * D.T + t) * D.S + i) * D.d;
}

double dot_in(const Dims& D, const void* a, int64_t oa, const void* b, int64_t ob) {
  double s = 0.0;
  for (int64_t c = 0; c < D.d; ++c) s += ld(a, D.dtype, oa + c) * ld(b, D.dtype, ob + c);
  return s;
}

// Forward for one query row (b, h, t): the plain joint-softmax definition.
// o[d] receives the normalised output; returns LSE.  scores is scratch space.
double row_forward(const Dims& D, const In& x, int64_t b, int64_t h, int64_t t, double* o,
                   std::vector<double>& scores) {
  const int64_t G = D.H / D.Hkv, g = h / G;
  const double sc = scale_of(D);
  const int64_t j0 = first_key(D, t), nseq = t - j0 + 1;
  scores.resize(static_cast<size_t>(nseq + D.S));
  const int64_t oq = off_q(D, b, h, t);
  for (int64_t j = j0; j <= t; ++j) scores[j - j0] = sc * dot_in(D, x.q, oq, x.k, off_kv(D, b, g, j));
  for (int64_t i = 0; i < D.S; ++i) scores[nseq + i] = sc * dot_in(D, x.q, oq, x.kd, off_dkv(D, b, g, t, i));
  double m = -std::numeric_limits<double>::infinity();
  for (double s : scores) m = std::max(m, s);
  double z = 0.0;
  for (int64_t c = 0; c < D.d; ++c) o[c] = 0.0;
  for (int64_t j = j0; j <= t; ++j) {
    double e = std::exp(scores[j - j0] - m);
    z += e;
    const int64_t ov = off_kv(D, b, g, j);
    for (int64_t c = 0; c < D.d; ++c) o[c] += e * ld(x.v, D.dtype, ov + c);
  }
  for (int64_t i = 0; i < D.S; ++i) {
    double e = std::exp(scores[nseq + i] - m);
    z += e;
    const int64_t ov = off_dkv(D, b, g, t, i);
    for (int64_t c = 0; c < D.d; ++c) o[c] += e * ld(x.vd, D.dtype, ov + c);
  }
  for (int64_t c = 0; c < D.d; ++c) o[c] /= z;
  return m + std::log(z);
}

// Per-row statistics the backward needs: LSE_t and D_t = dO_t . o_t.
void row_stats(const Dims& D, const In& x, int64_t b, int64_t h, int64_t t, double* lse, double* Dt,
               std::vector<double>& o, std::vector<double>& scores) {
  o.resize(static_cast<size_t>(D.d));
  *lse = row_forward(D, x, b, h, t, o.data(), scores);
  const int64_t oq = off_q(D, b, h, t);
  double s = 0.0;
  for (int64_t c = 0; c < D.d; ++c) s += ld(x.dout, D.dtype, oq + c) * o[c];
  *Dt = s;
}

// Backward, position part: for position (b, g, t) and each head h of group g,
// dq_t (sequence and depth terms), and the depth-slab gradients dkd_t, dvd_t.
// dq: [G, d]; dkd, dvd: [S, d] (accumulated over the G heads here).
void position_backward(const Dims& D, const In& x, int64_t b, int64_t g, int64_t t, double* dq,
                       double* dkd, double* dvd) {
  const int64_t G = D.H / D.Hkv;
  const double sc = scale_of(D);
  std::vector<double> o, scores;
  for (int64_t i = 0; i < D.S * D.d; ++i) dkd[i] = dvd[i] = 0.0;
  for (int64_t hh = 0; hh < G; ++hh) {
    const int64_t h = g * G + hh;
    double lse, Dt;
    row_stats(D, x, b, h, t, &lse, &Dt, o, scores);
    const int64_t oq = off_q(D, b, h, t);
    double* dqr = dq + hh * D.d;
    for (int64_t c = 0; c < D.d; ++c) dqr[c] = 0.0;
    const int64_t j0 = first_key(D, t);
    for (int64_t j = j0; j <= t; ++j) {
      const int64_t okv = off_kv(D, b, g, j);
      double p = std::exp(sc * dot_in(D, x.q, oq, x.k, okv) - lse);
      double dp = dot_in(D, x.dout, oq, x.v, okv);
      double ds = p * (dp - Dt);
      for (int64_t c = 0; c < D.d; ++c) dqr[c] += sc * ds * ld(x.k, D.dtype, okv + c);
    }
    for (int64_t i = 0; i < D.S; ++i) {
      const int64_t od = off_dkv(D, b, g, t, i);
      double p = std::exp(sc * dot_in(D, x.q, oq, x.kd, od) - lse);
      double dp = dot_in(D, x.dout, oq, x.vd, od);
      double ds = p * (dp - Dt);
      for (int64_t c = 0; c < D.d; ++c) {
        dqr[c] += sc * ds * ld(x.kd, D.dtype, od + c);
        dkd[i * D.d + c] += sc * ds * ld(x.q, D.dtype, oq + c);
        dvd[i * D.d + c] += p * ld(x.dout, D.dtype, oq + c);
      }
    }
  }
}

// Backward, key-column part: dk_j and dv_j for sequence key j of (b, g),
// summed over every visible row (h in g, t >= j).  lse/Dt: per-row statistics
// of group (b, g) laid out [G, T].
void key_backward(const Dims& D, const In& x, int64_t b, int64_t g, int64_t j, const double* lse,
                  const double* Dt, double* dk, double* dv) {
  const int64_t G = D.H / D.Hkv;
  const double sc = scale_of(D);
  const int64_t okv = off_kv(D, b, g, j);
  for (int64_t c = 0; c < D.d; ++c) dk[c] = dv[c] = 0.0;
  const int64_t t_end = D.seq_window > 0 ? std::min<int64_t>(D.T - 1, j + D.seq_window - 1) : D.T - 1;
  for (int64_t hh = 0; hh < G; ++hh) {
    const int64_t h = g * G + hh;
    for (int64_t t = j; t <= t_end; ++t) {
      const int64_t oq = off_q(D, b, h, t);
      double p = std::exp(sc * dot_in(D, x.q, oq, x.k, okv) - lse[hh * D.T + t]);
      double dp = dot_in(D, x.dout, oq, x.v, okv);
      double ds = p * (dp - Dt[hh * D.T + t]);
      for (int64_t c = 0; c < D.d; ++c) {
        dk[c] += sc * ds * ld(x.q, D.dtype, oq + c);
        dv[c] += p * ld(x.dout, D.dtype, oq + c);
      }
    }
  }
}

bool dims_ok(const Dims* D) {
  return D && D->B >= 0 && D->H > 0 && D->Hkv > 0 && D->H % D->Hkv == 0 && D->T >= 0 && D->S >= 0 &&
         D->d > 0 && (D->dtype == ORC_F64 || D->dtype == ORC_F32 || D->dtype == ORC_BF16);
}

}  // namespace

extern "C" {

// Number of host cores in this process's affinity mask.
int orc_cores() { return cores_available(); }

// Forward for a list of query rows (flat index r = (b*H + h)*T + t), or for
// every row when rows == nullptr (then n_rows is ignored and o is [B,H,T,d]).
// o: [n_rows, d] float64;  lse: [n_rows] float64.  Returns 0, or -1 on bad dims.
int orc_forward(const Dims* D, const void* q, const void* k, const void* v, const void* kd, const void* vd,
                const int64_t* rows, int64_t n_rows, double* o, double* lse) {
  if (!dims_ok(D)) return -1;
  const In x{q, k, v, kd, vd, nullptr};
  const int64_t n = rows ? n_rows : D->B * D->H * D->T;
  parallel_for(n, threads_for(*D), [&](int64_t idx) {
    const int64_t r = rows ? rows[idx] : idx;
    const int64_t t = r % D->T, bh = r / D->T, h = bh % D->H, b = bh / D->H;
    std::vector<double> scores;
    lse[idx] = row_forward(*D, x, b, h, t, o + idx * D->d, scores);
  });
  return 0;
}

// Backward, position part for a list of positions (flat p = (b*Hkv + g)*T + t),
// or for every position when pos == nullptr.
// dq: [n, G, d] (the G query heads of the position);  dkd, dvd: [n, S, d].
int orc_backward_positions(const Dims* D, const void* q, const void* k, const void* v, const void* kd,
                           const void* vd, const void* dout, const int64_t* pos, int64_t n_pos, double* dq,
                           double* dkd, double* dvd) {
  if (!dims_ok(D)) return -1;
  const In x{q, k, v, kd, vd, dout};
  const int64_t G = D->H / D->Hkv;
  const int64_t n = pos ? n_pos : D->B * D->Hkv * D->T;
  parallel_for(n, threads_for(*D), [&](int64_t idx) {
    const int64_t p = pos ? pos[idx] : idx;
    const int64_t t = p % D->T, bg = p / D->T, g = bg % D->Hkv, b = bg / D->Hkv;
    position_backward(*D, x, b, g, t, dq + idx * G * D->d, dkd + idx * D->S * D->d, dvd + idx * D->S * D->d);
  });
  return 0;
}

// Backward, key-column part for a list of sequence keys (flat p = (b*Hkv + g)*T + j),
// or for every key when keys == nullptr.  dk, dv: [n, d].
int orc_backward_keys(const Dims* D, const void* q, const void* k, const void* v, const void* kd,
                      const void* vd, const void* dout, const int64_t* keys, int64_t n_keys, double* dk,
                      double* dv) {
  if (!dims_ok(D)) return -1;
  const In x{q, k, v, kd, vd, dout};
  const int64_t G = D->H / D->Hkv;
  const int64_t n = keys ? n_keys : D->B * D->Hkv * D->T;
  const int nt = threads_for(*D);
  // Row statistics for every group that a requested key touches, from the
  // smallest requested key position onwards.
  const int64_t ngroups = D->B * D->Hkv;
  std::vector<int64_t> jmin(static_cast<size_t>(ngroups), D->T);
  for (int64_t idx = 0; idx < n; ++idx) {
    const int64_t p = keys ? keys[idx] : idx;
    const int64_t bg = p / D->T;
    jmin[bg] = std::min(jmin[bg], p % D->T);
  }
  std::vector<double> lse(static_cast<size_t>(ngroups * G * D->T), 0.0), Dt(lse.size(), 0.0);
  // Work items: (group, head-in-group, t) with t >= jmin[group].
  parallel_for(ngroups * G * D->T, nt, [&](int64_t w) {
    const int64_t t = w % D->T, gh = w / D->T, hh = gh % G, bg = gh / G;
    if (t < jmin[bg]) return;
    const int64_t b = bg / D->Hkv, g = bg % D->Hkv, h = g * G + hh;
    std::vector<double> o, scores;
    row_stats(*D, x, b, h, t, &lse[w], &Dt[w], o, scores);
  });
  parallel_for(n, nt, [&](int64_t idx) {
    const int64_t p = keys ? keys[idx] : idx;
    const int64_t j = p % D->T, bg = p / D->T, g = bg % D->Hkv, b = bg / D->Hkv;
    key_backward(*D, x, b, g, j, &lse[bg * G * D->T], &Dt[bg * G * D->T], dk + idx * D->d, dv + idx * D->d);
  });
  return 0;
}

}  // extern "C"
