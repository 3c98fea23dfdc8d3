// CPU oracle for the FP8 lightning indexer and its exact top-k selector.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct statement of what the
// indexer computes.  Only the test suite, the smoke check and the benchmark's CPU-baseline leg
// load it.  It shares no code, header, table or constant with the CUDA library, and the CUDA
// library never calls it.
//
// Every function follows the plain definition, in double precision, with no blocking, fusion
// or reordering:
//
//  * e4m3 decode -- OCP 8-bit floating point, E4M3FN variant (the format of the fp8 index
//    vectors in the TileLang deepseek_v32 README, "Lightning Indexer"; largest finite value
//    448 as noted in the FlashInfer MLA-decode discussion): 1 sign bit s, 4 exponent bits e
//    (bias 7), 3 mantissa bits m.  e > 0: (-1)^s 2^(e-7) (1 + m/8);  e = 0: (-1)^s 2^-6 (m/8);
//    s.1111.111 is NaN; there are no infinities.
//
//  * score -- Modular "sparse_index_fp8_sm100_prefill", the per-(token, key) logit formula, and
//    the TileLang README, "Lightning Indexer" (relu, weight by the per-(token, head) weight,
//    scale by the key's scale, sum over heads):
//        score[t, j] = k_scale[j] * sum_h relu( sum_d q[t,h,d] k[j,d] ) * w[t,h]
//    for j in the token's window [ks[t], ke[t]) clamped to [0, N] (the README's per-token
//    CuSeqLenKS / CuSeqLenKE bounds, clamped to seq_len_kv).  The dot product runs over d in
//    increasing order, the head sum over h in increasing order; k_scale multiplies the head sum.
//
//  * top-k -- TileLang README, "Top-k Selector": per query row, the k keys of largest score
//    within the window.  Ties are broken by the lower key index.  The selected key indices are
//    written in ascending order; a row whose window holds fewer than k keys is padded with -1
//    (the "-1 means no key" convention of the DeepSeek V4.1 sparse_attn_kernel page).  This is
//    done by a full sort of (score, index) pairs, never by a partial or radix method.
//
//  * key quantisation (the step that writes the fp8 index keys: TileLang README, "Lightning
//    Indexer", whose index vectors are FP8-quantized; 448 is the e4m3 maximum, FlashInfer MLA
//    decode discussion) -- per key row of D bf16 values x: s = max_j |x_j| / 448 (fp32
//    division), code_j = the e4m3 value nearest to x_j / s (fp32 division), ties to the even
//    code, magnitudes beyond 448 saturating to 448, the sign kept (also for a zero result).  A
//    row of zeros has s = 0 and all codes 0.  The nearest value is found by comparing against
//    every finite e4m3 magnitude (brute force).
//
//  * sparse attention over the selected keys (the step that consumes the indices: DeepSeek V4.1
//    sparse_attn_kernel page, and the TileLang README, "Sparse MLA Forward": attention is
//    evaluated only at the listed key positions, -1 entries are skipped) -- for query row t and
//    head h, with L the list idx[t, :] without its -1 entries (a key listed twice counts twice):
//        s_j      = scale * sum_d q[t,h,d] kv[j,d]                         (j in L)
//        o[t,h,:] = sum_j e^{s_j} kv[j,:] / ( sum_j e^{s_j} + e^{sink[h]} )
//    Each kv row is both key and value (the page's single kv tensor).  The optional per-head
//    sink adds e^{sink[h]} to the denominator only; without it the denominator is sum_j e^{s_j}.
//    An empty list gives o = 0.  Every exponent has the largest one (over the s_j and the sink)
//    subtracted first, which leaves the quotient unchanged and keeps e^x finite.  q and kv are
//    bf16 (exact in double).
//
//  * its gradients (TileLang README, "Sparse MLA Backward": delta = the row-wise product of the
//    output and its gradient; the softmax gradient P (dP - delta); dQ from dS and the listed
//    rows; dKV from dS and q plus P and dO, accumulated at the listed positions) -- for the loss
//    sum_{t,h,d} do[t,h,d] o[t,h,d] with do given (bf16), per row t and head h:
//        p_j = e^{s_j} / den,  p_sink = e^{sink[h]} / den      (den as in the forward)
//        dP_j = sum_d do[t,h,d] kv[j,d],   delta = sum_j p_j dP_j   (= do[t,h,:] . o[t,h,:])
//        ds_j = p_j (dP_j - delta)
//        dq[t,h,:]  = scale sum_j ds_j kv[j,:]
//        dkv[j,:]  += scale ds_j q[t,h,:] + p_j do[t,h,:]      (every listed occurrence of j)
//        dsink[h]  += -p_sink delta
//    Rows are taken in increasing t, list entries in list order, heads in increasing h.

// Build: g++ -O2 -std=c++17 -fPIC -shared (no -ffast-math: IEEE double semantics throughout).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <utility>
#include <vector>

namespace {

double e4m3_value(uint8_t code) {
  const int s = (code >> 7) & 1;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  if (e == 0xF && m == 0x7) return std::nan("");
  double mag;
  if (e == 0) {
    mag = std::ldexp(static_cast<double>(m) / 8.0, -6);
  } else {
    mag = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 7);
  }
  return s ? -mag : mag;
}

struct Table {
  double v[256];
  Table() {
    for (int c = 0; c < 256; ++c) v[c] = e4m3_value(static_cast<uint8_t>(c));
  }
};

const Table& table() {
  static const Table t;
  return t;
}

int64_t clamp64(int64_t x, int64_t lo, int64_t hi) { return x < lo ? lo : (x > hi ? hi : x); }

template <class F>
void parallel_rows(int64_t nrows, int nthreads, F&& body) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  if (nthreads == 1 || nrows < 2) {
    for (int64_t r = 0; r < nrows; ++r) body(r);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(nthreads);
  for (int i = 0; i < nthreads; ++i) {
    pool.emplace_back([&, i]() {
      // strided assignment: rows of very different length (causal windows) spread evenly
      for (int64_t r = i; r < nrows; r += nthreads) body(r);
    });
  }
  for (auto& th : pool) th.join();
}

// One query row: scores of the keys j in [lo, hi), written to out[j - lo].
void score_row(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale, int64_t t, int64_t lo,
               int64_t hi, int H, int D, double* out) {
  const double* tab = table().v;
  for (int64_t j = lo; j < hi; ++j) {
    double head_sum = 0.0;
    for (int h = 0; h < H; ++h) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d) {
        dot += tab[q[(t * H + h) * D + d]] * tab[k[j * D + d]];
      }
      const double relu = dot > 0.0 ? dot : 0.0;
      head_sum += relu * static_cast<double>(w[t * H + h]);
    }
    out[j - lo] = static_cast<double>(k_scale[j]) * head_sum;
  }
}

// Top-k of one row.  win[j - lo] is the score of key j, for j in [lo, hi).
template <class S>
void topk_row(const S* win, int64_t lo, int64_t hi, int topk, int32_t* out) {
  std::vector<std::pair<double, int64_t>> cand;  // (score, key index)
  cand.reserve(static_cast<size_t>(hi > lo ? hi - lo : 0));
  for (int64_t j = lo; j < hi; ++j) cand.emplace_back(static_cast<double>(win[j - lo]), j);
  // larger score first; equal scores: lower key index first (-0 and +0 compare equal)
  std::sort(cand.begin(), cand.end(), [](const std::pair<double, int64_t>& a, const std::pair<double, int64_t>& b) {
    if (a.first != b.first) return a.first > b.first;
    return a.second < b.second;
  });
  const int64_t take = std::min<int64_t>(topk, static_cast<int64_t>(cand.size()));
  std::vector<int64_t> sel;
  sel.reserve(static_cast<size_t>(take));
  for (int64_t i = 0; i < take; ++i) sel.push_back(cand[static_cast<size_t>(i)].second);
  std::sort(sel.begin(), sel.end());
  for (int i = 0; i < topk; ++i) out[i] = i < take ? static_cast<int32_t>(sel[static_cast<size_t>(i)]) : -1;
}

}  // namespace

// Nearest finite e4m3 code to y (a float, exact in double), ties to the even code, saturating.
static uint8_t e4m3_nearest(float y) {
  const uint8_t sign = std::signbit(y) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(y));
  int best = 0;
  double best_err = a;  // code 0 (value 0)
  for (int c = 1; c < 0x7F; ++c) {  // every finite non-negative code, in increasing value
    const double err = std::fabs(a - e4m3_value(static_cast<uint8_t>(c)));
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best = c;
      best_err = err;
    }
  }
  // beyond the largest finite value (448) every magnitude maps to it (the loop already picks
  // 0x7E for those: it is the nearest finite value)
  return static_cast<uint8_t>(sign | best);
}

extern "C" {

// out[c] = value of e4m3 code c (NaN for 0x7F and 0xFF).
void oracle_e4m3_table(double* out) {
  for (int c = 0; c < 256; ++c) out[c] = table().v[c];
}

// Window lengths of the listed rows: len[r] = max(0, clamp(ke[t]) - clamp(ks[t])), t = rows[r].
int oracle_window_lengths(const int32_t* ks, const int32_t* ke, int64_t T, int64_t N, const int64_t* rows,
                          int64_t nrows, int64_t* lo, int64_t* len) {
  if (!ks || !ke || !rows || !lo || !len || N < 0) return -1;
  for (int64_t r = 0; r < nrows; ++r) {
    if (rows[r] < 0 || rows[r] >= T) return -1;
    const int64_t a = clamp64(ks[rows[r]], 0, N), b = clamp64(ke[rows[r]], 0, N);
    lo[r] = a;
    len[r] = b > a ? b - a : 0;
  }
  return 0;
}

// Scores of the query rows listed in `rows` (nrows entries, each in [0, T)).  Row r's window
// [lo, hi) (ks/ke clamped to [0, N]) is written compactly: out[offsets[r] + (j - lo)] is the
// score of key j.  The caller sizes offsets from oracle_window_lengths.
// Returns 0, or -1 on a bad argument.
int oracle_index_score(const uint8_t* q, const float* w, const uint8_t* k, const float* k_scale, const int32_t* ks,
                       const int32_t* ke, int64_t T, int64_t N, int H, int D, const int64_t* rows, int64_t nrows,
                       const int64_t* offsets, double* out, int nthreads) {
  if (!q || !w || !k || !k_scale || !ks || !ke || !rows || !offsets || !out || T < 0 || N < 0 || H < 1 || D < 1)
    return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= T) return -1;
  parallel_rows(nrows, nthreads, [&](int64_t r) {
    const int64_t t = rows[r];
    const int64_t lo = clamp64(ks[t], 0, N);
    const int64_t hi = clamp64(ke[t], 0, N);
    score_row(q, w, k, k_scale, t, lo, hi, H, D, out + offsets[r]);
  });
  return 0;
}

// Top-k over compact score rows: row r holds len[r] scores at scores[offsets[r] + i] for the
// keys lo[r] + i.  idx is [nrows, topk] of absolute key indices.
// Returns 0, or -1 on a bad argument or a NaN score.
int oracle_topk_compact(const double* scores, const int64_t* offsets, const int64_t* lo, const int64_t* len,
                        int64_t nrows, int topk, int32_t* idx, int nthreads) {
  if (!scores || !offsets || !lo || !len || !idx || topk < 1) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    for (int64_t i = 0; i < len[r]; ++i)
      if (std::isnan(scores[offsets[r] + i])) return -1;
  parallel_rows(nrows, nthreads, [&](int64_t r) {
    topk_row(scores + offsets[r], lo[r], lo[r] + len[r], topk, idx + r * topk);
  });
  return 0;
}

// Top-k of nrows score rows (row r is scores + r * row_stride, window [ks[r], ke[r]) clamped to
// [0, N]).  idx is [nrows, topk].  Returns 0, or -1 on a bad argument or a NaN in a window.
int oracle_topk_f64(const double* scores, int64_t row_stride, const int32_t* ks, const int32_t* ke, int64_t nrows,
                    int64_t N, int topk, int32_t* idx, int nthreads) {
  if (!scores || !ks || !ke || !idx || topk < 1 || N < 0) return -1;
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t lo = clamp64(ks[r], 0, N), hi = clamp64(ke[r], 0, N);
    for (int64_t j = lo; j < hi; ++j)
      if (std::isnan(scores[r * row_stride + j])) return -1;
  }
  parallel_rows(nrows, nthreads, [&](int64_t r) {
    const int64_t lo = clamp64(ks[r], 0, N), hi = clamp64(ke[r], 0, N);
    topk_row(scores + r * row_stride + lo, lo, hi, topk, idx + r * topk);
  });
  return 0;
}

// The same selection over fp32 score rows (used on a GPU-produced logits buffer: only the
// in-window entries are read, so whatever lies outside the window is never looked at).
int oracle_topk_f32(const float* scores, int64_t row_stride, const int32_t* ks, const int32_t* ke, int64_t nrows,
                    int64_t N, int topk, int32_t* idx, int nthreads) {
  if (!scores || !ks || !ke || !idx || topk < 1 || N < 0) return -1;
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t lo = clamp64(ks[r], 0, N), hi = clamp64(ke[r], 0, N);
    for (int64_t j = lo; j < hi; ++j)
      if (std::isnan(scores[r * row_stride + j])) return -1;
  }
  parallel_rows(nrows, nthreads, [&](int64_t r) {
    const int64_t lo = clamp64(ks[r], 0, N), hi = clamp64(ke[r], 0, N);
    topk_row(scores + r * row_stride + lo, lo, hi, topk, idx + r * topk);
  });
  return 0;
}

// Quantises N rows of D bf16 values (bit patterns): codes [N, D] and per-row scales [N].
int oracle_quantize_rows(const uint16_t* x_bf16, int64_t N, int64_t D, uint8_t* codes, float* scale) {
  for (int64_t r = 0; r < N; ++r) {
    std::vector<float> x(static_cast<size_t>(D));
    for (int64_t j = 0; j < D; ++j) {
      const uint32_t bits = static_cast<uint32_t>(x_bf16[r * D + j]) << 16;  // bf16 -> fp32 exactly
      std::memcpy(&x[static_cast<size_t>(j)], &bits, 4);
    }
    float m = 0.0f;
    for (float v : x) m = std::max(m, std::fabs(v));
    const float s = m / 448.0f;
    scale[r] = s;
    for (int64_t j = 0; j < D; ++j) {
      codes[r * D + j] = m == 0.0f ? 0 : e4m3_nearest(x[static_cast<size_t>(j)] / s);
    }
  }
  return 0;
}

// Sparse attention of T query rows over the listed keys (see the header): q bf16 bits
// [T, H, D], kv bf16 bits [N, D], sink [H] or null, idx [T, K] (-1 or a key in [0, N)),
// out [T, H, D] in double.  Returns -1 (nothing written) if an index is out of range.
int oracle_sparse_attn(const uint16_t* q_bf16, const uint16_t* kv_bf16, const float* sink, const int32_t* idx,
                       int64_t T, int64_t N, int64_t H, int64_t D, int64_t K, double scale, double* out,
                       int nthreads) {
  if (!q_bf16 || !kv_bf16 || !idx || !out || T < 0 || N < 0 || H < 1 || D < 1 || K < 0) return -1;
  for (int64_t i = 0; i < T * K; ++i)
    if (idx[i] < -1 || idx[i] >= N) return -1;
  auto bf16 = [](uint16_t b) {
    const uint32_t bits = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return static_cast<double>(f);
  };
  parallel_rows(T, nthreads, [&](int64_t t) {
    std::vector<int64_t> list;
    for (int64_t i = 0; i < K; ++i)
      if (idx[t * K + i] >= 0) list.push_back(idx[t * K + i]);
    for (int64_t h = 0; h < H; ++h) {
      double* o = out + (t * H + h) * D;
      for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
      if (list.empty()) continue;
      std::vector<double> s(list.size());
      for (size_t a = 0; a < list.size(); ++a) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += bf16(q_bf16[(t * H + h) * D + d]) * bf16(kv_bf16[list[a] * D + d]);
        s[a] = scale * dot;
      }
      double m = s[0];
      for (double v : s) m = std::max(m, v);
      if (sink) m = std::max(m, static_cast<double>(sink[h]));
      double den = sink ? std::exp(static_cast<double>(sink[h]) - m) : 0.0;
      for (size_t a = 0; a < list.size(); ++a) {
        const double e = std::exp(s[a] - m);
        den += e;
        for (int64_t d = 0; d < D; ++d) o[d] += e * bf16(kv_bf16[list[a] * D + d]);
      }
      for (int64_t d = 0; d < D; ++d) o[d] /= den;
    }
  });
  return 0;
}

// Gradients of the sparse attention (see the header): do bf16 bits [T, H, D]; dq [T, H, D],
// dkv [N, D] and dsink [H] (when sink is given; may be null otherwise) in double, overwritten.
// Returns -1 (nothing written) if an index is out of range.  Rows are independent for dq; dkv
// is summed per key over the rows that list it, in increasing row and list position.
int oracle_sparse_attn_bwd(const uint16_t* q_bf16, const uint16_t* kv_bf16, const float* sink, const int32_t* idx,
                           const uint16_t* do_bf16, int64_t T, int64_t N, int64_t H, int64_t D, int64_t K,
                           double scale, double* dq, double* dkv, double* dsink, int nthreads) {
  if (!q_bf16 || !kv_bf16 || !idx || !do_bf16 || !dq || !dkv || T < 0 || N < 0 || H < 1 || D < 1 || K < 0) return -1;
  for (int64_t i = 0; i < T * K; ++i)
    if (idx[i] < -1 || idx[i] >= N) return -1;
  auto bf16 = [](uint16_t b) {
    const uint32_t bits = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &bits, 4);
    return static_cast<double>(f);
  };
  auto qv = [&](int64_t t, int64_t h, int64_t d) { return bf16(q_bf16[(t * H + h) * D + d]); };
  auto dov = [&](int64_t t, int64_t h, int64_t d) { return bf16(do_bf16[(t * H + h) * D + d]); };
  auto kvv = [&](int64_t j, int64_t d) { return bf16(kv_bf16[j * D + d]); };
  auto score = [&](int64_t t, int64_t h, int64_t j) {
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += qv(t, h, d) * kvv(j, d);
    return scale * dot;
  };
  auto dprob = [&](int64_t t, int64_t h, int64_t j) {
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += dov(t, h, d) * kvv(j, d);
    return dot;
  };
  // pass 1, per row: the softmax's shift and denominator, delta and the sink's weight, and dq
  std::vector<double> shift(static_cast<size_t>(T * H)), den(static_cast<size_t>(T * H)),
      delta(static_cast<size_t>(T * H)), psink(static_cast<size_t>(T * H));
  parallel_rows(T, nthreads, [&](int64_t t) {
    std::vector<int64_t> list;
    for (int64_t i = 0; i < K; ++i)
      if (idx[t * K + i] >= 0) list.push_back(idx[t * K + i]);
    for (int64_t h = 0; h < H; ++h) {
      double* g = dq + (t * H + h) * D;
      for (int64_t d = 0; d < D; ++d) g[d] = 0.0;
      const size_t th = static_cast<size_t>(t * H + h);
      shift[th] = 0.0;
      den[th] = 1.0;
      delta[th] = 0.0;
      psink[th] = 0.0;
      if (list.empty()) continue;
      std::vector<double> s(list.size()), dp(list.size());
      for (size_t a = 0; a < list.size(); ++a) {
        s[a] = score(t, h, list[a]);
        dp[a] = dprob(t, h, list[a]);
      }
      double m = s[0];
      for (double v : s) m = std::max(m, v);
      if (sink) m = std::max(m, static_cast<double>(sink[h]));
      double z = sink ? std::exp(static_cast<double>(sink[h]) - m) : 0.0;
      for (size_t a = 0; a < list.size(); ++a) z += std::exp(s[a] - m);
      double dl = 0.0;
      for (size_t a = 0; a < list.size(); ++a) dl += std::exp(s[a] - m) / z * dp[a];
      for (size_t a = 0; a < list.size(); ++a) {
        const double ds = std::exp(s[a] - m) / z * (dp[a] - dl);
        for (int64_t d = 0; d < D; ++d) g[d] += scale * ds * kvv(list[a], d);
      }
      shift[th] = m;
      den[th] = z;
      delta[th] = dl;
      psink[th] = sink ? std::exp(static_cast<double>(sink[h]) - m) / z : 0.0;
    }
  });
  // pass 2, per key: its occurrences in increasing (row, list position), every head
  std::vector<std::vector<std::pair<int64_t, int64_t>>> occ(static_cast<size_t>(N));
  for (int64_t t = 0; t < T; ++t)
    for (int64_t i = 0; i < K; ++i)
      if (idx[t * K + i] >= 0) occ[static_cast<size_t>(idx[t * K + i])].push_back({t, i});
  parallel_rows(N, nthreads, [&](int64_t j) {
    double* g = dkv + j * D;
    for (int64_t d = 0; d < D; ++d) g[d] = 0.0;
    for (const auto& o : occ[static_cast<size_t>(j)]) {
      const int64_t t = o.first;
      for (int64_t h = 0; h < H; ++h) {
        const size_t th = static_cast<size_t>(t * H + h);
        const double pj = std::exp(score(t, h, j) - shift[th]) / den[th];
        const double ds = pj * (dprob(t, h, j) - delta[th]);
        for (int64_t d = 0; d < D; ++d) g[d] += scale * ds * qv(t, h, d) + pj * dov(t, h, d);
      }
    }
  });
  if (dsink) {
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int64_t t = 0; t < T; ++t) acc += -psink[static_cast<size_t>(t * H + h)] * delta[static_cast<size_t>(t * H + h)];
      dsink[h] = acc;
    }
  }
  return 0;
}

// The encoder alone, for the tests' pins.
int oracle_e4m3_encode(const float* y, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = e4m3_nearest(y[i]);
  return 0;
}

}  // extern "C"
