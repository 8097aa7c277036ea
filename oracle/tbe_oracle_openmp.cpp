// TBE oracle, OpenMP form -- TEST INFRASTRUCTURE ONLY (the timed CPU baseline).
//
// The oracle's pooled forward and its backward with exactly one Adagrad update
// per touched row, with the loops spread over the host's cores: the forward in
// parallel over bags; the backward groups the lookups by row with a parallel
// stable sort (a scatter into key-range buckets that keeps lookup order, then
// a stable sort of each bucket by key) and updates the rows of the run map in
// parallel.  Every number is formed by the oracle's own helpers (included
// below), in the oracle's order: a bag sums its rows in ascending lookup
// order, a row sums its lookups' gradient rows in ascending lookup order, so
// both entry points give bit for bit what oracle_forward and
// oracle_backward_rowwise_adagrad give (tests/test_oracle_openmp.py).  Only
// the bench's CPU baseline and the tests load this library.

#include "tbe_oracle.cpp"

#include <omp.h>

namespace {

// One valid lookup of the backward: its linear key, its position in
// indices[] and its bag within its table.
struct Lookup {
  uint32_t key;
  uint32_t bag;
  int64_t pos;
};

// The valid lookups sorted by (key, position): the lookups scattered in
// position order into nbk key-range buckets (per-thread counts, then each
// thread writes its own position range), then each bucket sorted stably by
// key.
std::vector<Lookup> sorted_lookups(const Problem& p) {
  const int64_t nb = static_cast<int64_t>(p.T) * p.B;
  const int64_t n_used = p.off(nb);
  const uint64_t total_E = static_cast<uint64_t>(p.hash_base[p.T]);
  const int P = omp_get_max_threads();
  const int nbk = 64 * P;
  auto bucket_of = [&](uint64_t key) { return static_cast<int>(key * nbk / total_E); };
  // lookup i: key (or none), bag; the table of position i from the bags
  std::vector<uint32_t> key(static_cast<size_t>(n_used));
  std::vector<uint32_t> bag(static_cast<size_t>(n_used));
  std::vector<uint8_t> ok(static_cast<size_t>(n_used), 0);
#pragma omp parallel for schedule(dynamic, 256)
  for (int64_t g = 0; g < nb; ++g) {
    const int t = static_cast<int>(g / p.B);
    for (int64_t i = p.off(g); i < p.off(g + 1); ++i) {
      const int64_t r = p.idx(i);
      if (!p.valid(t, r)) continue;
      key[i] = static_cast<uint32_t>(p.hash_base[t] + r);
      bag[i] = static_cast<uint32_t>(g % p.B);
      ok[i] = 1;
    }
  }
  // counts of bucket k in position chunk c, then their starts in (k, c) order
  std::vector<int64_t> cnt(static_cast<size_t>(P) * nbk, 0);
  auto chunk = [&](int c, int64_t* lo, int64_t* hi) {
    *lo = n_used * c / P;
    *hi = n_used * (c + 1) / P;
  };
#pragma omp parallel for schedule(static, 1)
  for (int c = 0; c < P; ++c) {
    int64_t lo, hi;
    chunk(c, &lo, &hi);
    int64_t* my = cnt.data() + static_cast<size_t>(c) * nbk;
    for (int64_t i = lo; i < hi; ++i)
      if (ok[i]) ++my[bucket_of(key[i])];
  }
  std::vector<int64_t> start(static_cast<size_t>(P) * nbk);
  std::vector<int64_t> bk_first(static_cast<size_t>(nbk) + 1);
  int64_t run = 0;
  for (int k = 0; k < nbk; ++k) {
    bk_first[k] = run;
    for (int c = 0; c < P; ++c) {
      start[static_cast<size_t>(c) * nbk + k] = run;
      run += cnt[static_cast<size_t>(c) * nbk + k];
    }
  }
  bk_first[nbk] = run;
  std::vector<Lookup> out(static_cast<size_t>(run));
#pragma omp parallel for schedule(static, 1)
  for (int c = 0; c < P; ++c) {
    int64_t lo, hi;
    chunk(c, &lo, &hi);
    int64_t* at = start.data() + static_cast<size_t>(c) * nbk;
    for (int64_t i = lo; i < hi; ++i)
      if (ok[i]) out[at[bucket_of(key[i])]++] = Lookup{key[i], bag[i], i};
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int k = 0; k < nbk; ++k)
    std::stable_sort(out.begin() + bk_first[k], out.begin() + bk_first[k + 1],
                     [](const Lookup& a, const Lookup& b) { return a.key < b.key; });
  return out;
}

}  // namespace

extern "C" {

int oracle_omp_threads(void) { return omp_get_max_threads(); }

// Threads of the parallel regions that follow (n > 0).
void oracle_omp_set_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
}

// As oracle_forward, the bags in parallel.
int oracle_omp_forward(int T, int B, const int64_t* D_offsets, const int64_t* hash_base,
                       const int64_t* w_offsets, const void* weights, int index_bits,
                       const void* indices, const void* offsets, int64_t n, const float* psw,
                       int mean, int wtype, float* out) {
  Problem p{T, B, D_offsets, hash_base, w_offsets, index_bits, indices, offsets, n, psw};
  if (!offsets_ok(p)) return ORACLE_EINVAL;
  if (wtype < 0 || wtype > 2) return ORACLE_EINVAL;
  const WeightArray W{const_cast<void*>(weights), wtype};
  const int64_t sumD = D_offsets[T];
  const int64_t nb = static_cast<int64_t>(T) * B;
#pragma omp parallel
  {
    std::vector<int64_t> rows;
    std::vector<float> coef;
#pragma omp for schedule(dynamic, 64)
    for (int64_t bag = 0; bag < nb; ++bag) {
      const int t = static_cast<int>(bag / B);
      const int64_t b = bag % B;
      const int D = static_cast<int>(p.D(t));
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

// As oracle_backward_rowwise_adagrad, the rows of the run map in parallel
// (each row is updated by one thread, from its lookups in ascending order).
int oracle_omp_backward(int T, int B, const int64_t* D_offsets, const int64_t* hash_base,
                        const int64_t* w_offsets, int index_bits, const void* indices,
                        const void* offsets, int64_t n, const float* psw, const float* grad_out,
                        int mean, int wtype, int elementwise, float lr, float eps,
                        void* weights, float* momentum) {
  Problem p{T, B, D_offsets, hash_base, w_offsets, index_bits, indices, offsets, n, psw};
  if (!offsets_ok(p)) return ORACLE_EINVAL;
  if (wtype < 0 || wtype > 2) return ORACLE_EINVAL;
  if (hash_base[T] <= 0 || static_cast<uint64_t>(hash_base[T]) > 0xffffffffull)
    return ORACLE_EINVAL;
  const WeightArray W{weights, wtype};
  const int64_t sumD = D_offsets[T];
  const std::vector<Lookup> s = sorted_lookups(p);
  const int64_t m = static_cast<int64_t>(s.size());
  // run starts: positions whose key differs from the one before
  std::vector<int64_t> runs;
  for (int64_t i = 0; i < m; ++i)
    if (i == 0 || s[i].key != s[i - 1].key) runs.push_back(i);
  runs.push_back(m);
  const int64_t R = static_cast<int64_t>(runs.size()) - 1;
#pragma omp parallel
  {
    std::vector<const float*> gp;
    std::vector<float> coef;
    std::vector<double> bs;
    std::vector<double> g;
#pragma omp for schedule(dynamic, 16)
    for (int64_t j = 0; j < R; ++j) {
      const uint64_t key = s[runs[j]].key;
      const int t = table_of_key(p, key);
      const int D = static_cast<int>(p.D(t));
      const int64_t r = static_cast<int64_t>(key) - hash_base[t];
      gp.clear();
      coef.clear();
      bs.clear();
      for (int64_t k = runs[j]; k < runs[j + 1]; ++k) {
        const Lookup& c = s[k];
        gp.push_back(grad_out + static_cast<int64_t>(c.bag) * sumD + D_offsets[t]);
        coef.push_back(psw ? psw[c.pos] : 1.0f);
        bs.push_back(p.mean_scale(static_cast<int64_t>(t) * B + c.bag));
      }
      g.assign(D, 0.0);
      sum_run_gradient(static_cast<int64_t>(gp.size()), D, gp.data(), coef.data(), g.data(),
                       mean ? bs.data() : nullptr);
      const int64_t w0 = w_offsets[t] + r * D;
      if (elementwise)
        elementwise_adagrad(D, g.data(), lr, eps, W, w0, momentum + w0);
      else
        rowwise_adagrad(D, g.data(), lr, eps, W, w0, momentum + key);
    }
  }
  return ORACLE_OK;
}

}  // extern "C"
