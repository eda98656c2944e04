// CPU oracle for exact Top-K over ragged FP32 score rows.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg may load this library.  It shares no code with
// the CUDA selector: no headers, no helpers, no constants.
//
// What it follows (sources are web pages about "Sample-Guided Exact Top-K
// Selection for Long-Context Sparse Attention", Tencent HPC-Ops):
//
//  * The set contract: codexqa.cn article "几何平均快 1.55 倍，但短行采样会输：
//    腾讯怎么测精确 Top-K", section "什么叫精确，时间怎么量".  Indices are
//    distinct and inside the valid prefix.  When the row length exceeds K the
//    set holds exactly K indices and its smallest score is not below the
//    largest score left out; boundary ties may be broken either way; output
//    order is free; there is no floating-point tolerance.  When the row length
//    is at most K every valid index is returned and the free slots hold the
//    contract's sentinel (read here as -1).
//  * "Exact" means the same set a full sort gives: PaperDaily walkthrough
//    "腾讯|长上下文稀疏注意力前K精确选择", section 问题二 (the final set equals
//    the exact baseline).  So the selection below is the plain definition: a
//    library selection (std::nth_element) under the order "larger score first,
//    then smaller index", which makes the oracle's own tie choice deterministic.
//  * The sampled thresholds: PaperDaily section 问题二 (Fig. 4 stage 1 and 2;
//    fixed-stride sample of the current row proposes a provisional tau0 and a
//    nested, wider tau1; C(tau) counts the full row's scores that reach tau;
//    C(tau0) >= K continues to refinement, else tau1, else exact recovery) and
//    the codexqa.cn section "采样不是处处都该开" (defaults: stride 128, primary
//    target 1.5K candidates, secondary 1.75K).  The rank rule that turns a
//    candidate target T into a sample rank is not printed; the reading used
//    here is r = ceil(T * n_s / len) clamped to [1, n_s], with samples at
//    positions 0, s, 2s, ... below len and n_s = ceil(len / s).
//
//  * The indexer scores that feed the selector: eq. (1) of the xllm-io
//    review of LiteTopK, section "核心公式" (see oracle_index_scores).
//
// All comparisons are plain C++ float comparisons (no bit tricks).  NaN is not
// a supported input.
//
// Row lengths outside [0, N_alloc] are clamped into that range, which is the
// behaviour the library under test documents for its own API.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

int64_t clamp_len(int32_t raw, int64_t n_alloc) {
  int64_t v = raw;
  if (v < 0) v = 0;
  if (v > n_alloc) v = n_alloc;
  return v;
}

// Runs fn(row_begin, row_end) over [0, M) split into contiguous blocks.
void parallel_rows(int64_t M, int threads, const std::function<void(int64_t, int64_t)>& fn) {
  if (threads <= 0) {
    threads = (int)std::thread::hardware_concurrency();
    if (threads <= 0) threads = 1;
  }
  if (M <= 0) return;
  if (threads > M) threads = (int)M;
  if (threads == 1) {
    fn(0, M);
    return;
  }
  // Interleave small blocks so ragged row costs spread over the threads.
  const int64_t block = 4;
  std::vector<std::thread> pool;
  pool.reserve(threads);
  for (int t = 0; t < threads; ++t) {
    pool.emplace_back([&, t]() {
      for (int64_t b = (int64_t)t * block; b < M; b += (int64_t)threads * block) {
        fn(b, std::min(M, b + block));
      }
    });
  }
  for (auto& th : pool) th.join();
}

// Index order of the oracle: higher score first; equal scores by lower index.
struct Before {
  const float* v;
  bool operator()(int32_t a, int32_t b) const {
    if (v[a] > v[b]) return true;
    if (v[b] > v[a]) return false;
    return a < b;
  }
};

}  // namespace

extern "C" {

// Exact Top-K per row.  out is [M][K] int32.  For len > K the K chosen indices
// are written in ascending index order (ordering is for comparison only; the
// contract leaves it free).  For len <= K the row holds 0..len-1 followed by
// K-len sentinels (-1).  Returns 0, or -1 on bad arguments.
int oracle_topk(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                int32_t K, int32_t* out, int threads) {
  if (M < 0 || N_alloc < 0 || K < 1) return -1;
  if (M > 0 && (!scores || !row_lens || !out)) return -1;
  parallel_rows(M, threads, [&](int64_t r0, int64_t r1) {
    std::vector<int32_t> idx;
    for (int64_t r = r0; r < r1; ++r) {
      const float* v = scores + r * N_alloc;
      int32_t* o = out + r * (int64_t)K;
      const int64_t L = clamp_len(row_lens[r], N_alloc);
      if (L <= K) {
        for (int64_t i = 0; i < K; ++i) o[i] = (i < L) ? (int32_t)i : -1;
        continue;
      }
      idx.resize((size_t)L);
      for (int64_t i = 0; i < L; ++i) idx[(size_t)i] = (int32_t)i;
      std::nth_element(idx.begin(), idx.begin() + K, idx.end(), Before{v});
      std::sort(idx.begin(), idx.begin() + K);
      std::memcpy(o, idx.data(), sizeof(int32_t) * (size_t)K);
    }
  });
  return 0;
}

// Contract checker, independent of oracle_topk.  row_err[r] receives:
//   0 ok
//   1 an index outside [0, len) that is not a sentinel slot
//   2 duplicate index
//   3 len > K and a sentinel (-1) appears (count of valid indices != K)
//   4 len > K and min(selected) < max(unselected)
//   5 len <= K and the valid indices are not exactly {0..len-1}
//   6 len <= K and the number of -1 sentinels is not K - len
// Returns the number of rows with a nonzero code, or -1 on bad arguments.
int64_t oracle_check(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                     int32_t K, const int32_t* out, int32_t* row_err, int threads) {
  if (M < 0 || N_alloc < 0 || K < 1) return -1;
  if (M > 0 && (!scores || !row_lens || !out || !row_err)) return -1;
  parallel_rows(M, threads, [&](int64_t r0, int64_t r1) {
    std::vector<uint8_t> seen;
    for (int64_t r = r0; r < r1; ++r) {
      const float* v = scores + r * N_alloc;
      const int32_t* o = out + r * (int64_t)K;
      const int64_t L = clamp_len(row_lens[r], N_alloc);
      seen.assign((size_t)L, 0);
      int32_t err = 0;
      int64_t n_valid = 0, n_sent = 0;
      for (int64_t i = 0; i < K && !err; ++i) {
        const int32_t x = o[i];
        if (x == -1) {
          ++n_sent;
          continue;
        }
        if (x < 0 || (int64_t)x >= L) {
          err = 1;
          break;
        }
        if (seen[(size_t)x]) {
          err = 2;
          break;
        }
        seen[(size_t)x] = 1;
        ++n_valid;
      }
      if (!err) {
        if (L > K) {
          if (n_sent != 0 || n_valid != K) {
            err = 3;
          } else {
            // min over the selected set vs max over the rest, as floats.
            bool have_sel = false, have_rest = false;
            float min_sel = 0.f, max_rest = 0.f;
            for (int64_t i = 0; i < L; ++i) {
              if (seen[(size_t)i]) {
                if (!have_sel || v[i] < min_sel) min_sel = v[i];
                have_sel = true;
              } else {
                if (!have_rest || v[i] > max_rest) max_rest = v[i];
                have_rest = true;
              }
            }
            if (have_sel && have_rest && min_sel < max_rest) err = 4;
          }
        } else {
          if (n_valid != L) err = 5;
          else if (n_sent != (int64_t)K - L) err = 6;
        }
      }
      row_err[r] = err;
    }
  });
  int64_t bad = 0;
  for (int64_t r = 0; r < M; ++r) bad += (row_err[r] != 0);
  return bad;
}

// For rows with len > K: kth[r] = K-th largest score, kth1[r] = (K+1)-th
// largest, tied[r] = 1 when they are equal as floats (the boundary is tied and
// several index sets are correct).  Rows with len <= K get tied = 0 and NaN in
// both value slots.
int oracle_boundary(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                    int32_t K, float* kth, float* kth1, uint8_t* tied, int threads) {
  if (M < 0 || N_alloc < 0 || K < 1) return -1;
  if (M > 0 && (!scores || !row_lens || !kth || !kth1 || !tied)) return -1;
  parallel_rows(M, threads, [&](int64_t r0, int64_t r1) {
    std::vector<float> vals;
    for (int64_t r = r0; r < r1; ++r) {
      const float* v = scores + r * N_alloc;
      const int64_t L = clamp_len(row_lens[r], N_alloc);
      if (L <= K) {
        kth[r] = NAN;
        kth1[r] = NAN;
        tied[r] = 0;
        continue;
      }
      vals.assign(v, v + L);
      // Largest first: position K-1 holds the K-th largest, position K the
      // (K+1)-th.
      std::nth_element(vals.begin(), vals.begin() + K, vals.end(), std::greater<float>());
      const float b = vals[(size_t)K];
      const float a = *std::min_element(vals.begin(), vals.begin() + K);
      kth[r] = a;
      kth1[r] = b;
      tied[r] = (a > b) ? 0 : 1;
    }
  });
  return 0;
}

// Sample-guided thresholds and the path a row takes, by the pages' stage
// definitions (see header).  target0/target1 are the candidate targets in
// elements (1.5K = 3072 and 1.75K = 3584 at K = 2048).  For each row:
//   tau[2r]   = tau0, the r0-th largest sample (r0 from target0)
//   tau[2r+1] = tau1, the r1-th largest sample (r1 from target1)
//   cnt[2r]   = C(tau0) = #{ i < len : v[i] >= tau0 }
//   cnt[2r+1] = C(tau1)
//   rank[2r], rank[2r+1] = r0, r1
//   path[r]: 0 len <= K (sentinel rows), 1 len < sample_min_len (exact,
//            no sampling), 2 C(tau0) >= K, 3 C(tau0) < K <= C(tau1),
//            4 C(tau1) < K (exact whole-row recovery).
// Rows on paths 0 and 1 get NaN thresholds, zero counts and zero ranks.
int oracle_thresholds(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                      int32_t K, int32_t stride, int32_t target0, int32_t target1,
                      int64_t sample_min_len, float* tau, int64_t* cnt, int64_t* rank,
                      int32_t* path, int threads) {
  if (M < 0 || N_alloc < 0 || K < 1 || stride < 1 || target0 < 1 || target1 < target0) return -1;
  if (M > 0 && (!scores || !row_lens || !tau || !cnt || !rank || !path)) return -1;
  parallel_rows(M, threads, [&](int64_t r0, int64_t r1) {
    std::vector<float> samp;
    for (int64_t r = r0; r < r1; ++r) {
      const float* v = scores + r * N_alloc;
      const int64_t L = clamp_len(row_lens[r], N_alloc);
      tau[2 * r] = NAN;
      tau[2 * r + 1] = NAN;
      cnt[2 * r] = cnt[2 * r + 1] = 0;
      rank[2 * r] = rank[2 * r + 1] = 0;
      if (L <= K) {
        path[r] = 0;
        continue;
      }
      if (L < sample_min_len) {
        path[r] = 1;
        continue;
      }
      samp.clear();
      for (int64_t i = 0; i < L; i += stride) samp.push_back(v[i]);
      const int64_t ns = (int64_t)samp.size();  // == ceil(L / stride)
      const int64_t targets[2] = {target0, target1};
      float t[2];
      for (int j = 0; j < 2; ++j) {
        int64_t rk = (targets[j] * ns + L - 1) / L;  // ceil(T * n_s / len)
        if (rk < 1) rk = 1;
        if (rk > ns) rk = ns;
        std::vector<float> s2 = samp;
        std::nth_element(s2.begin(), s2.begin() + (rk - 1), s2.end(), std::greater<float>());
        t[j] = s2[(size_t)(rk - 1)];
        rank[2 * r + j] = rk;
      }
      int64_t c0 = 0, c1 = 0;
      for (int64_t i = 0; i < L; ++i) {
        c0 += (v[i] >= t[0]);
        c1 += (v[i] >= t[1]);
      }
      tau[2 * r] = t[0];
      tau[2 * r + 1] = t[1];
      cnt[2 * r] = c0;
      cnt[2 * r + 1] = c1;
      path[r] = (c0 >= K) ? 2 : (c1 >= K) ? 3 : 4;
    }
  });
  return 0;
}

// Indexer scores (the score stage that produces the rows the selector
// reads), the plain definition of eq. (1) in the xllm-io review of LiteTopK,
// section "核心公式":
//   I[t][s] = sum over heads j of w[t][j] * ReLU( dot(q[t][j][:], k[s][:]) ).
// q is [T][H][D] and k is [S][D], both bfloat16 given as raw 16-bit patterns
// (a bfloat16 is the upper half of an IEEE binary32, so widening is exact);
// w is [T][H] float.  Everything is accumulated in double.  For each of the
// n requested pairs (ts[i], ss[i]) writes value[i] = I and magnitude[i] =
// sum_j |w[t][j]| * sum_d |q[t][j][d] * k[s][d]|, the scale against which a
// lower-precision evaluation's rounding error is measured.  Returns 0, or -1
// on bad arguments.
static double bf16_to_double(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return (double)f;
}

int oracle_index_scores(const uint16_t* q, const uint16_t* k, const float* w, int64_t T, int64_t S,
                        int64_t H, int64_t D, const int64_t* ts, const int64_t* ss, int64_t n,
                        double* value, double* magnitude, int threads) {
  if (T < 0 || S < 0 || H < 1 || D < 1 || n < 0) return -1;
  if (n > 0 && (!q || !k || !w || !ts || !ss || !value || !magnitude)) return -1;
  for (int64_t i = 0; i < n; ++i)
    if (ts[i] < 0 || ts[i] >= T || ss[i] < 0 || ss[i] >= S) return -1;
  parallel_rows(n, threads, [&](int64_t i0, int64_t i1) {
    for (int64_t i = i0; i < i1; ++i) {
      const int64_t t = ts[i], sidx = ss[i];
      double acc = 0.0, mag = 0.0;
      for (int64_t j = 0; j < H; ++j) {
        double dot = 0.0, adot = 0.0;
        for (int64_t d = 0; d < D; ++d) {
          const double prod = bf16_to_double(q[(t * H + j) * D + d]) * bf16_to_double(k[sidx * D + d]);
          dot += prod;
          adot += std::fabs(prod);
        }
        const double wj = (double)w[t * H + j];
        acc += wj * (dot > 0.0 ? dot : 0.0);
        mag += std::fabs(wj) * adot;
      }
      value[i] = acc;
      magnitude[i] = mag;
    }
  });
  return 0;
}

// The optional ordered output.  The contract leaves the order of a Top-K
// result free (codexqa.cn section "什么叫精确，时间怎么量"; PaperDaily
// section 问题二: the result is a set, not sorted by score); an ordered
// result is the same set listed by score, largest first, equal scores by
// smaller index first, with the -1 sentinel slots last.  in_idx and out_idx
// are [M][K] int32 (they may be the same array); every entry of in_idx is -1
// or an index below row_lens[r] (clamped), else the call returns -1 without
// writing that row's output.  Returns 0, or -1 on bad arguments or a bad
// index.
int oracle_order(const float* scores, const int32_t* row_lens, int64_t M, int64_t N_alloc,
                 int32_t K, const int32_t* in_idx, int32_t* out_idx, int threads) {
  if (M < 0 || N_alloc < 0 || K < 1) return -1;
  if (M > 0 && (!scores || !row_lens || !in_idx || !out_idx)) return -1;
  std::vector<uint8_t> bad((size_t)(M > 0 ? M : 0), 0);
  parallel_rows(M, threads, [&](int64_t r0, int64_t r1) {
    std::vector<int32_t> idx;
    for (int64_t r = r0; r < r1; ++r) {
      const float* v = scores + r * N_alloc;
      const int32_t* in = in_idx + r * (int64_t)K;
      const int64_t L = clamp_len(row_lens[r], N_alloc);
      idx.clear();
      for (int64_t i = 0; i < K; ++i) {
        if (in[i] == -1) continue;
        if (in[i] < 0 || (int64_t)in[i] >= L) {
          bad[(size_t)r] = 1;
          break;
        }
        idx.push_back(in[i]);
      }
      if (bad[(size_t)r]) continue;
      std::sort(idx.begin(), idx.end(), Before{v});
      int32_t* o = out_idx + r * (int64_t)K;
      for (int64_t i = 0; i < K; ++i) o[i] = i < (int64_t)idx.size() ? idx[(size_t)i] : -1;
    }
  });
  for (int64_t r = 0; r < M; ++r)
    if (bad[(size_t)r]) return -1;
  return 0;
}

// Hardware threads this library uses when threads <= 0 is passed.
int oracle_default_threads(void) {
  int t = (int)std::thread::hardware_concurrency();
  return t > 0 ? t : 1;
}

}  // extern "C"
