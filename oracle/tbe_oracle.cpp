// TBE oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU statement of what the Table Batched
// Embedding (TBE) hot path computes.  Only tests/, the package smoke check and
// the bench's cpu_baseline / reference arm may load this library; the product
// path never does.  It shares no code, header, table or helper with the CUDA
// library: every conversion and formula below is written out here on its own.
//
// Sources (pages; section, equation or table named, no code copied):
//  * "Modernizing Table Batched Embeddings with FBTriton" (yuxiaoba.github.io,
//    English page), section "Forward: keep a narrowly specialized path beside
//    the general one": each bag sums the rows it indexes; fp16 weights are
//    accumulated in wider precision.  The oracle accumulates in double.
//  * same page, section "Backward: invert 'which rows did this sample use?'":
//    lookups are regrouped into runs, one per unique (table,row); every run's
//    gradients are summed and the row is updated exactly once.
//  * same page, section "Fusion boundaries are also engineering interfaces":
//    per-sample weights scale each contribution before grouping.
//  * "HugeCTR DistributedSlotSparseEmbeddingHash backward" (eqicode.com),
//    steps 1-5 of the update and the Adagrad kernel: stable sort of
//    (row, sample) pairs, run starts with a sentinel, accumulator updated
//    first and the weight step using the new accumulator with eps outside the
//    square root.  The row-wise form replaces the element-wise accumulator
//    increment g_d^2 by the row mean (1/D) sum_d g_d^2; the element-wise
//    form itself (one accumulator per weight element, at the weight's own
//    flat position) is offered beside it.
//
//  * same HugeCTR page, the combiner note (sum, or mean = the sum kernel then
//    a scaling kernel) and the mean backward kernel: with mean pooling a
//    bag's gradient is multiplied by 1/L, L the bag's number of lookups by
//    the row offsets, when L > 1, before the regrouping.  The forward scaling
//    kernel is not printed: the oracle takes the plainest reading, the pooled
//    sum times the same factor.
//
// Readings where the pages are silent:
//  * bags are table-major: bag (t,b) has id t*B+b, offsets has T*B+1 entries;
//  * a lookup whose row is outside [0, E_t) contributes nothing (skipped);
//  * weights are fp16 (or bf16, or fp32), rounded to nearest-even from the
//    double result; every type is pooled in double (the page pools fp32
//    weights in fp64 and 16-bit ones in fp32: both are within the double
//    sum's rounding of the exact sum);
//  * momentum is fp32, rounded from the double sum m_old + mean_d(g_d^2)
//    (element-wise: m_old_d + g_d^2 per element).
//
// Parity pins for every function live in tests/test_oracle_*.py.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <vector>

namespace {

// ---------------------------------------------------------------- fp16 bits
// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double half_bits_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int expo = (h >> 10) & 0x1f;
  const int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = std::ldexp(static_cast<double>(frac), -24);  // subnormal: frac * 2^-24
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(1024 + frac), expo - 25);
  }
  return sign ? -v : v;
}

// Round a double to the nearest binary16, ties to even.
uint16_t double_to_half_bits(double x) {
  if (std::isnan(x)) return 0x7e00;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  double a = std::fabs(x);
  if (a == 0.0) return sign;
  // Largest finite half is 65504; halfway to the next binade step is 65520.
  if (a >= 65520.0) return sign | 0x7c00;
  if (a < std::ldexp(1.0, -14)) {
    // Subnormal range: the unit is 2^-24.  q == 1024 lands on the smallest
    // normal, whose bit pattern is exactly 0x0400.
    double q = std::nearbyint(std::ldexp(a, 24));
    return sign | static_cast<uint16_t>(q);
  }
  int e2;
  std::frexp(a, &e2);          // a = f * 2^e2, f in [0.5, 1)
  int e = e2 - 1;              // a in [2^e, 2^(e+1))
  double q = std::nearbyint(std::ldexp(a, 10 - e));  // in [1024, 2048]
  if (q == 2048.0) {
    q = 1024.0;
    e += 1;
  }
  if (e + 15 >= 31) return sign | 0x7c00;
  return sign | static_cast<uint16_t>(((e + 15) << 10) | (static_cast<int>(q) - 1024));
}

// --------------------------------------------------------------- bf16 bits
// bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits -- the
// upper half of a binary32.
double bf16_bits_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int expo = (h >> 7) & 0xff;
  const int frac = h & 0x7f;
  double v;
  if (expo == 0) {
    v = std::ldexp(static_cast<double>(frac), -133);  // subnormal: frac * 2^-133
  } else if (expo == 255) {
    v = frac ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(128 + frac), expo - 134);
  }
  return sign ? -v : v;
}

// Round a double to the nearest bfloat16, ties to even.
uint16_t double_to_bf16_bits(double x) {
  if (std::isnan(x)) return 0x7fc0;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (a == 0.0) return sign;
  if (a < std::ldexp(1.0, -126)) {
    // subnormal range, unit 2^-133; q == 128 is the smallest normal 0x0080
    const double q = std::nearbyint(std::ldexp(a, 133));
    return sign | static_cast<uint16_t>(q);
  }
  int e2;
  std::frexp(a, &e2);
  int e = e2 - 1;                                    // a in [2^e, 2^(e+1))
  double q = std::nearbyint(std::ldexp(a, 7 - e));   // in [128, 256]
  if (q == 256.0) {
    q = 128.0;
    e += 1;
  }
  if (e + 127 >= 255) return sign | 0x7f80;          // overflow to infinity
  return sign | static_cast<uint16_t>(((e + 127) << 7) | (static_cast<int>(q) - 128));
}

// A flat weight array of one element type (wtype): 0 fp16 and 1 bf16 (16-bit
// patterns), 2 fp32.  Elements are read exactly as doubles and written
// rounded to nearest even in the array's own type (fp32 by the language's
// double-to-float conversion, which rounds to nearest even).
struct WeightArray {
  void* base;
  int wtype;
  double get(int64_t i) const {
    if (wtype == 2) return static_cast<double>(static_cast<const float*>(base)[i]);
    const uint16_t h = static_cast<const uint16_t*>(base)[i];
    return wtype == 1 ? bf16_bits_to_double(h) : half_bits_to_double(h);
  }
  void set(int64_t i, double x) const {
    if (wtype == 2) {
      static_cast<float*>(base)[i] = static_cast<float>(x);
      return;
    }
    static_cast<uint16_t*>(base)[i] = wtype == 1 ? double_to_bf16_bits(x) : double_to_half_bits(x);
  }
};

int64_t load_int(const void* p, int bits, int64_t i) {
  if (bits == 32) return static_cast<const int32_t*>(p)[i];
  return static_cast<const int64_t*>(p)[i];
}

// Pool one bag: out[d] = (float) (scale * sum_k coef_k * row_k[d]), summed in
// double in ascending k; row k starts at element row_start[k] of W.
// coef == nullptr means every coefficient is 1.
void pool_rows(int64_t L, int D, const WeightArray& W, const int64_t* row_start,
               const float* coef, float* out, double scale = 1.0) {
  for (int d = 0; d < D; ++d) {
    double s = 0.0;
    for (int64_t k = 0; k < L; ++k) {
      const double w = coef ? static_cast<double>(coef[k]) : 1.0;
      s += w * W.get(row_start[k] + d);
    }
    out[d] = static_cast<float>(s * scale);
  }
}

// Sum one run's gradient: g[d] = sum_k coef_k * bag_scale_k * grad_k[d] in
// double, ascending k (bag_scale == nullptr: every factor is 1).
void sum_run_gradient(int64_t SL, int D, const float* const* grads, const float* coef,
                      double* g, const double* bag_scale = nullptr) {
  for (int d = 0; d < D; ++d) {
    double s = 0.0;
    for (int64_t k = 0; k < SL; ++k) {
      double w = coef ? static_cast<double>(coef[k]) : 1.0;
      if (bag_scale) w *= bag_scale[k];
      s += w * static_cast<double>(grads[k][d]);
    }
    g[d] = s;
  }
}


// Exact row-wise Adagrad on one row, given its summed gradient g[0..D):
//   m <- m + (1/D) sum_d g_d^2          (stored as fp32)
//   w_d <- w_d - lr * g_d / (sqrt(m) + eps)   (stored in the weight type,
//                                              nearest-even); the row starts
//                                              at element w0 of W
void rowwise_adagrad(int D, const double* g, float lr, float eps, const WeightArray& W,
                     int64_t w0, float* m) {
  double ss = 0.0;
  for (int d = 0; d < D; ++d) ss += g[d] * g[d];
  const float m_new = static_cast<float>(static_cast<double>(*m) + ss / static_cast<double>(D));
  *m = m_new;
  const double denom = std::sqrt(static_cast<double>(m_new)) + static_cast<double>(eps);
  for (int d = 0; d < D; ++d) {
    const double w_old = W.get(w0 + d);
    W.set(w0 + d, w_old - static_cast<double>(lr) * g[d] / denom);
  }
}

struct Problem {
  int T, B;
  const int64_t* D_offsets;   // [T+1] cumulative widths
  const int64_t* hash_base;   // [T+1] cumulative row counts
  const int64_t* w_offsets;   // [T+1] element offset of each table in the flat weights
  int index_bits;             // 32 or 64; offsets share the index type
  const void* indices;        // [n]
  const void* offsets;        // [T*B+1]
  int64_t n;
  const float* psw;           // [n] or nullptr

  int64_t D(int t) const { return D_offsets[t + 1] - D_offsets[t]; }
  int64_t E(int t) const { return hash_base[t + 1] - hash_base[t]; }
  int64_t off(int64_t bag) const { return load_int(offsets, index_bits, bag); }
  int64_t idx(int64_t i) const { return load_int(indices, index_bits, i); }
  bool valid(int t, int64_t r) const { return r >= 0 && r < E(t); }
  // Mean pooling's factor for bag `bag`: 1/L when its L lookups (by the
  // offsets, rows out of range included) number more than one, else 1.
  double mean_scale(int64_t bag) const {
    const int64_t L = off(bag + 1) - off(bag);
    return L > 1 ? 1.0 / static_cast<double>(L) : 1.0;
  }
};

// Offsets must satisfy 0 = o[0] <= o[1] <= ... <= o[T*B] <= n; lookups at or
// after o[T*B] belong to no bag.
bool offsets_ok(const Problem& p) {
  const int64_t nb = static_cast<int64_t>(p.T) * p.B;
  if (p.off(0) != 0 || p.off(nb) > p.n) return false;
  for (int64_t i = 0; i < nb; ++i)
    if (p.off(i) > p.off(i + 1)) return false;
  return true;
}

struct Contribution {
  int64_t pos;   // lookup position in indices[]
  uint32_t bag;  // b, the bag within its table
  double mean_scale;  // the bag's mean-pooling factor
};

// One std::map entry per touched (table,row), keyed by the linear key
// hash_base[t] + row; each entry lists its lookups in ascending position.
std::map<uint64_t, std::vector<Contribution>> group_by_row(const Problem& p) {
  std::map<uint64_t, std::vector<Contribution>> runs;
  for (int t = 0; t < p.T; ++t) {
    for (int64_t b = 0; b < p.B; ++b) {
      const int64_t bag = static_cast<int64_t>(t) * p.B + b;
      for (int64_t i = p.off(bag); i < p.off(bag + 1); ++i) {
        const int64_t r = p.idx(i);
        if (!p.valid(t, r)) continue;
        runs[static_cast<uint64_t>(p.hash_base[t] + r)].push_back(
            {i, static_cast<uint32_t>(b), p.mean_scale(bag)});
      }
    }
  }
  return runs;
}

int table_of_key(const Problem& p, uint64_t key) {
  for (int t = 0; t < p.T; ++t)
    if (static_cast<int64_t>(key) < p.hash_base[t + 1]) return t;
  return -1;
}

}  // namespace

extern "C" {

// Status codes returned by every entry point.
enum { ORACLE_OK = 0, ORACLE_EINVAL = 1 };

double oracle_half_to_double(uint16_t h) { return half_bits_to_double(h); }
uint16_t oracle_double_to_half(double x) { return double_to_half_bits(x); }
double oracle_bf16_to_double(uint16_t h) { return bf16_bits_to_double(h); }
uint16_t oracle_double_to_bf16(double x) { return double_to_bf16_bits(x); }

// Pooled forward over every bag: out[b, D_offsets[t] + d] for all t, b, d.
// out is fp32 row-major [B, D_offsets[T]].
int oracle_forward(int T, int B, const int64_t* D_offsets, const int64_t* hash_base,
                   const int64_t* w_offsets, const void* weights, int index_bits,
                   const void* indices, const void* offsets, int64_t n, const float* psw,
                   int mean, int wtype, float* out) {
  Problem p{T, B, D_offsets, hash_base, w_offsets, index_bits, indices, offsets, n, psw};
  if (!offsets_ok(p)) return ORACLE_EINVAL;
  if (wtype < 0 || wtype > 2) return ORACLE_EINVAL;
  const WeightArray W{const_cast<void*>(weights), wtype};
  const int64_t sumD = D_offsets[T];
  std::vector<int64_t> rows;
  std::vector<float> coef;
  for (int t = 0; t < T; ++t) {
    const int D = static_cast<int>(p.D(t));
    for (int64_t b = 0; b < B; ++b) {
      const int64_t bag = static_cast<int64_t>(t) * B + b;
      rows.clear();
      coef.clear();
      for (int64_t i = p.off(bag); i < p.off(bag + 1); ++i) {
        const int64_t r = p.idx(i);
        if (!p.valid(t, r)) continue;
        rows.push_back(w_offsets[t] + r * D);
        coef.push_back(psw ? psw[i] : 1.0f);
      }
      pool_rows(static_cast<int64_t>(rows.size()), D, W, rows.data(), coef.data(),
                out + b * sumD + D_offsets[t], mean ? p.mean_scale(bag) : 1.0);
    }
  }
  return ORACLE_OK;
}

// Pooled forward of bags whose rows were gathered beforehand: bag j pools
// rows[k*D .. k*D+D) for k in [bag_off[j], bag_off[j+1]), scaled by coef[k]
// (coef may be null).  out is [nbags, D].  Used to check sampled bags of
// workloads too large to hold on the host.
int oracle_pool_gathered(int64_t nbags, int D, const int64_t* bag_off, const uint16_t* rows,
                         const float* coef, float* out) {
  const WeightArray W{const_cast<uint16_t*>(rows), 0};
  std::vector<int64_t> rp;
  for (int64_t j = 0; j < nbags; ++j) {
    const int64_t L = bag_off[j + 1] - bag_off[j];
    if (L < 0) return ORACLE_EINVAL;
    rp.resize(L);
    for (int64_t k = 0; k < L; ++k) rp[k] = (bag_off[j] + k) * D;
    pool_rows(L, D, W, rp.data(), coef ? coef + bag_off[j] : nullptr, out + j * D);
  }
  return ORACLE_OK;
}

// Preprocessing: every valid lookup i of bag (t,b) becomes the pair
// (key = hash_base[t] + row, bag = b).  Pairs are stable-sorted by key and
// run-length encoded.  Outputs (caller sizes them for n entries, R+1 for rs):
//   sorted_keys[n_valid], sorted_bags[n_valid], sorted_pos[n_valid],
//   unique_keys[R], run_starts[R+1] with run_starts[R] = n_valid.
// *n_valid_out and *R_out receive the counts.
int oracle_preprocess(int T, int B, const int64_t* hash_base, int index_bits,
                      const void* indices, const void* offsets, int64_t n,
                      uint32_t* sorted_keys, uint32_t* sorted_bags, int64_t* sorted_pos,
                      uint32_t* unique_keys, int64_t* run_starts, int64_t* n_valid_out,
                      int64_t* R_out) {
  // D_offsets and w_offsets are not needed here.
  Problem p{T, B, nullptr, hash_base, nullptr, index_bits, indices, offsets, n, nullptr};
  if (!offsets_ok(p)) return ORACLE_EINVAL;
  struct Entry {
    uint32_t key;
    uint32_t bag;
    int64_t pos;
  };
  std::vector<Entry> e;
  e.reserve(n);
  for (int t = 0; t < T; ++t)
    for (int64_t b = 0; b < B; ++b) {
      const int64_t bag = static_cast<int64_t>(t) * B + b;
      for (int64_t i = p.off(bag); i < p.off(bag + 1); ++i) {
        const int64_t r = p.idx(i);
        if (!p.valid(t, r)) continue;
        e.push_back({static_cast<uint32_t>(hash_base[t] + r), static_cast<uint32_t>(b), i});
      }
    }
  std::stable_sort(e.begin(), e.end(),
                   [](const Entry& a, const Entry& b) { return a.key < b.key; });
  int64_t R = 0;
  for (size_t i = 0; i < e.size(); ++i) {
    sorted_keys[i] = e[i].key;
    sorted_bags[i] = e[i].bag;
    sorted_pos[i] = e[i].pos;
    if (i == 0 || e[i].key != e[i - 1].key) {
      unique_keys[R] = e[i].key;
      run_starts[R] = static_cast<int64_t>(i);
      ++R;
    }
  }
  run_starts[R] = static_cast<int64_t>(e.size());
  *n_valid_out = static_cast<int64_t>(e.size());
  *R_out = R;
  return ORACLE_OK;
}

// Summed gradient of every touched row, in ascending key order:
// g[j*maxD + d] = sum over the run's lookups i of psw_i * s_i * grad_out[b_i, D_offsets[t]+d]
// (double; s_i the bag's mean-pooling factor when mean != 0, else 1).  keys[j] receives the run's linear key.  Sized for n runs.
int oracle_row_gradients(int T, int B, const int64_t* D_offsets, const int64_t* hash_base,
                         int index_bits, const void* indices, const void* offsets, int64_t n,
                         const float* psw, const float* grad_out, int mean, int maxD,
                         uint32_t* keys, double* g, int64_t* R_out) {
  Problem p{T, B, D_offsets, hash_base, nullptr, index_bits, indices, offsets, n, psw};
  if (!offsets_ok(p)) return ORACLE_EINVAL;
  const int64_t sumD = D_offsets[T];
  auto runs = group_by_row(p);
  int64_t j = 0;
  std::vector<const float*> gp;
  std::vector<float> coef;
  std::vector<double> bs;  // the lookups' bag factors (mean pooling)
  for (const auto& kv : runs) {
    const int t = table_of_key(p, kv.first);
    const int D = static_cast<int>(p.D(t));
    gp.clear();
    coef.clear();
    bs.clear();
    for (const Contribution& c : kv.second) {
      gp.push_back(grad_out + static_cast<int64_t>(c.bag) * sumD + D_offsets[t]);
      coef.push_back(psw ? psw[c.pos] : 1.0f);
      bs.push_back(c.mean_scale);
    }
    keys[j] = static_cast<uint32_t>(kv.first);
    std::fill(g + j * maxD, g + (j + 1) * maxD, 0.0);
    sum_run_gradient(static_cast<int64_t>(gp.size()), D, gp.data(), coef.data(), g + j * maxD,
                     mean ? bs.data() : nullptr);
    ++j;
  }
  *R_out = j;
  return ORACLE_OK;
}

// Element-wise Adagrad on one row (the HugeCTR page's Adagrad kernel: the
// accumulator is per weight element), given its summed gradient g[0..D):
//   m_d <- m_d + g_d^2                          (stored as fp32)
//   w_d <- w_d - lr * g_d / (sqrt(m_d) + eps)   (stored in the weight type)
void elementwise_adagrad(int D, const double* g, float lr, float eps, const WeightArray& W,
                         int64_t w0, float* m) {
  for (int d = 0; d < D; ++d) {
    const float m_new = static_cast<float>(static_cast<double>(m[d]) + g[d] * g[d]);
    m[d] = m_new;
    const double denom = std::sqrt(static_cast<double>(m_new)) + static_cast<double>(eps);
    const double w_old = W.get(w0 + d);
    W.set(w0 + d, w_old - static_cast<double>(lr) * g[d] / denom);
  }
}

// Backward with exactly one Adagrad update per touched row, in place on
// weights (16-bit patterns, flat) and momentum: row-wise, fp32 [hash_base[T]];
// element-wise (elementwise != 0), fp32 laid out like the weights.
int oracle_backward_rowwise_adagrad(int T, int B, const int64_t* D_offsets,
                                    const int64_t* hash_base, const int64_t* w_offsets,
                                    int index_bits, const void* indices, const void* offsets,
                                    int64_t n, const float* psw, const float* grad_out,
                                    int mean, int wtype, int elementwise, float lr, float eps,
                                    void* weights, float* momentum) {
  Problem p{T, B, D_offsets, hash_base, w_offsets, index_bits, indices, offsets, n, psw};
  if (!offsets_ok(p)) return ORACLE_EINVAL;
  if (wtype < 0 || wtype > 2) return ORACLE_EINVAL;
  const WeightArray W{weights, wtype};
  const int64_t sumD = D_offsets[T];
  auto runs = group_by_row(p);
  std::vector<const float*> gp;
  std::vector<float> coef;
  std::vector<double> bs;  // the lookups' bag factors (mean pooling)
  std::vector<double> g;
  for (const auto& kv : runs) {
    const int t = table_of_key(p, kv.first);
    const int D = static_cast<int>(p.D(t));
    const int64_t r = static_cast<int64_t>(kv.first) - hash_base[t];
    gp.clear();
    coef.clear();
    bs.clear();
    for (const Contribution& c : kv.second) {
      gp.push_back(grad_out + static_cast<int64_t>(c.bag) * sumD + D_offsets[t]);
      coef.push_back(psw ? psw[c.pos] : 1.0f);
      bs.push_back(c.mean_scale);
    }
    g.assign(D, 0.0);
    sum_run_gradient(static_cast<int64_t>(gp.size()), D, gp.data(), coef.data(), g.data(),
                     mean ? bs.data() : nullptr);
    const int64_t w0 = w_offsets[t] + r * D;
    if (elementwise)
      elementwise_adagrad(D, g.data(), lr, eps, W, w0, momentum + w0);
    else
      rowwise_adagrad(D, g.data(), lr, eps, W, w0, momentum + kv.first);
  }
  return ORACLE_OK;
}

// Backward restricted to selected rows, for workloads too large to update on
// the host.  sel_keys[j] is a linear key; w_rows[j*maxD ..] holds that row's
// fp16 weights and m_rows[j] its momentum on entry, the updated values on
// exit.  All lookups are scanned; only those of selected keys contribute.
// contrib_out[j] (nullable) receives each selected row's run length.
int oracle_backward_selected(int T, int B, const int64_t* D_offsets, const int64_t* hash_base,
                             int index_bits, const void* indices, const void* offsets, int64_t n,
                             const float* psw, const float* grad_out, int mean, float lr,
                             float eps, int64_t nsel, const uint32_t* sel_keys, int maxD,
                             uint16_t* w_rows,
                             float* m_rows, int64_t* contrib_out) {
  Problem p{T, B, D_offsets, hash_base, nullptr, index_bits, indices, offsets, n, psw};
  if (!offsets_ok(p)) return ORACLE_EINVAL;
  const int64_t sumD = D_offsets[T];
  std::map<uint64_t, int64_t> slot;
  for (int64_t j = 0; j < nsel; ++j) slot[sel_keys[j]] = j;
  std::vector<std::vector<Contribution>> lists(nsel);
  for (int t = 0; t < T; ++t)
    for (int64_t b = 0; b < B; ++b) {
      const int64_t bag = static_cast<int64_t>(t) * B + b;
      for (int64_t i = p.off(bag); i < p.off(bag + 1); ++i) {
        const int64_t r = p.idx(i);
        if (!p.valid(t, r)) continue;
        auto it = slot.find(static_cast<uint64_t>(hash_base[t] + r));
        if (it != slot.end())
          lists[it->second].push_back({i, static_cast<uint32_t>(b), p.mean_scale(bag)});
      }
    }
  std::vector<const float*> gp;
  std::vector<float> coef;
  std::vector<double> bs;  // the lookups' bag factors (mean pooling)
  std::vector<double> g;
  for (int64_t j = 0; j < nsel; ++j) {
    if (contrib_out) contrib_out[j] = static_cast<int64_t>(lists[j].size());
    if (lists[j].empty()) continue;  // untouched rows keep their values
    const int t = table_of_key(p, sel_keys[j]);
    if (t < 0) return ORACLE_EINVAL;
    const int D = static_cast<int>(p.D(t));
    gp.clear();
    coef.clear();
    bs.clear();
    for (const Contribution& c : lists[j]) {
      gp.push_back(grad_out + static_cast<int64_t>(c.bag) * sumD + D_offsets[t]);
      coef.push_back(psw ? psw[c.pos] : 1.0f);
      bs.push_back(c.mean_scale);
    }
    g.assign(D, 0.0);
    sum_run_gradient(static_cast<int64_t>(gp.size()), D, gp.data(), coef.data(), g.data(),
                     mean ? bs.data() : nullptr);
    rowwise_adagrad(D, g.data(), lr, eps, WeightArray{w_rows, 0}, j * maxD, m_rows + j);
  }
  return ORACLE_OK;
}

// Offset repair, the reading used when the checker runs in repair mode:
// o'[0] = 0 and, for i >= 1, o'[i] = max(o'[i-1], clamp(o[i], 0, n)).
// The result is non-decreasing and inside [0, n]; lookups at or after
// o'[T*B] belong to no bag.  Returns the number of entries that changed.
int64_t oracle_repair_offsets(int index_bits, const void* offsets_in, int64_t nb1, int64_t n,
                              int64_t* offsets_out) {
  int64_t changed = 0;
  int64_t prev = 0;
  for (int64_t i = 0; i < nb1; ++i) {
    const int64_t o = load_int(offsets_in, index_bits, i);
    int64_t v;
    if (i == 0) {
      v = 0;
    } else {
      v = std::min<int64_t>(std::max<int64_t>(o, 0), n);
      v = std::max(v, prev);
    }
    if (v != o) ++changed;
    offsets_out[i] = v;
    prev = v;
  }
  return changed;
}

}  // extern "C"
