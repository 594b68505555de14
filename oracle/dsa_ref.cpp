// CPU oracle of the DeepSeek Sparse Attention (DSA) hot path, in C++ --
// TEST INFRASTRUCTURE.
//
// Only the tests, __graft_entry__.smoke() and bench.py's CPU-baseline / oracle
// legs load this library (through oracle/cpp.py).  It shares no code, header
// or constant with the CUDA library: it includes only the C++ standard
// library.  Plain loops in double precision; the only parallelism is one query
// row per task on std::thread workers, so every row is computed exactly as
// the definitions read.  Inputs are the exact values of the bf16 / fp32
// tensors the GPU path receives, widened to double by the caller.
//
// Sources (pages; titles abbreviated as below):
//  [DSA-32K] "CANN&TorchTitan: DeepSeek-V3.2 32k long-sequence pretraining on
//            Ascend" -- section "DSA fused ops / SparseLightningIndexerGradKLLoss"
//            (Lightning Indexer forward formula; Sparse Flash Attention forward
//            formula; KL loss; dI; dW / dq~ / dK~ formulas) and section
//            "SparseFlashAttentionGrad" (gather, softmax recompute, dP, dS, dQ,
//            dK, dV formulas).
//  [HP-CP]   "CP context parallel guide" -- section "DSA CP" (query rows of a
//            shard at global positions, replicated key side) and the
//            load_balance note (the mask is built from K's length).
//  [NPU-ops] "CANN/torchtitan-npu fused-operator adaptation" -- section "DSA":
//            the indexer's top-k indices drive the sparse attention.
//
// Readings where the pages are silent (the same as the Python oracle's):
// scores over all causal keys s <= pos(t), no extra scale; top-k order value
// descending then index ascending, -0.0 == +0.0, output ascending, -1 padding;
// one index set per token shared by every head; V = the first d_v columns of
// the kv row; softmax_max / softmax_sum over the scaled logits with natural
// exp; the KL target sums the per-head probabilities over heads then
// L1-normalises over the selected keys; the loss sums over tokens; 0 log 0 = 0;
// ReLU'(0) = 0; D = sum_e dY * O; dK and dV of the shared kv row add into one
// dKV; dQ and dK carry `scale`.
//
// Accumulations across query rows (dkv, dk_I) are atomic double additions, so
// their order, and their last bits, may vary from run to run; the loss is
// summed over rows in row order.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// Runs f(row) for row in [0, n) on `threads` workers, rows handed out one at
// a time (causal rows differ widely in cost).
template <class F>
void for_rows(long long n, int threads, F f) {
  if (threads < 1) threads = 1;
  if (threads > n) threads = (int)(n > 0 ? n : 1);
  std::atomic<long long> next{0};
  auto work = [&]() {
    for (;;) {
      const long long r = next.fetch_add(1);
      if (r >= n) break;
      f(r);
    }
  };
  if (threads == 1) {
    work();
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t) pool.emplace_back(work);
  for (auto& th : pool) th.join();
}

void atomic_add(double* p, double v) { std::atomic_ref<double>(*p).fetch_add(v); }

// The valid (>= 0) entries of one index row, in slot order.
std::vector<long long> selected(const int32_t* idx_row, long long k) {
  std::vector<long long> sel;
  for (long long i = 0; i < k; ++i)
    if (idx_row[i] >= 0) sel.push_back(idx_row[i]);
  return sel;
}

// Logits of token r for head h over the selected keys: scale * q[r,h,:] . kv[b,s,:]
void logits(const double* qh, const double* kvb, long long d_qk, const std::vector<long long>& sel,
            double scale, std::vector<double>& out) {
  out.resize(sel.size());
  for (size_t i = 0; i < sel.size(); ++i) {
    const double* kr = kvb + sel[i] * d_qk;
    double acc = 0.0;
    for (long long d = 0; d < d_qk; ++d) acc += qh[d] * kr[d];
    out[i] = scale * acc;
  }
}

}  // namespace

extern "C" {

// [DSA-32K] Lightning Indexer forward: I[t, s] = sum_j w[t, j] ReLU(q_I[t, j, :] . k_I[s, :])
// for every causal key s <= pos(t) of the row's batch; -inf elsewhere.
// q_I [B*S_q, H_I, d_I], k_I [B, S_k, d_I], w [B*S_q, H_I], pos [B*S_q] ->
// scores [B*S_q, S_k].
void dsa_ref_indexer_scores(long long B, long long S_q, long long S_k, long long H_I,
                            long long d_I, const double* q_I, const double* k_I, const double* w,
                            const long long* pos, double* scores, int threads) {
  for_rows(B * S_q, threads, [&](long long r) {
    const long long b = r / S_q, p = pos[r];
    double* out = scores + r * S_k;
    for (long long s = 0; s < S_k; ++s) {
      if (s > p) {
        out[s] = kNegInf;
        continue;
      }
      const double* ks = k_I + (b * S_k + s) * d_I;
      double I = 0.0;
      for (long long j = 0; j < H_I; ++j) {
        const double* qj = q_I + (r * H_I + j) * d_I;
        double dot = 0.0;
        for (long long d = 0; d < d_I; ++d) dot += qj[d] * ks[d];
        I += w[r * H_I + j] * (dot > 0.0 ? dot : 0.0);
      }
      out[s] = I;
    }
  });
}

// [DSA-32K] the top-k positions of each token: among s <= pos(t), order by
// value descending then index ascending (doubles compare -0.0 equal to +0.0),
// keep the first min(k, pos(t)+1), write them in ascending index order, pad -1.
void dsa_ref_topk(long long rows, long long S_k, long long k, const double* scores,
                  const long long* pos, int32_t* idx, int threads) {
  for_rows(rows, threads, [&](long long r) {
    const double* row = scores + r * S_k;
    const long long n = pos[r] + 1;
    std::vector<long long> order(n);
    for (long long s = 0; s < n; ++s) order[s] = s;
    std::stable_sort(order.begin(), order.end(),
                     [row](long long a, long long c) { return row[a] > row[c]; });
    const long long keep = std::min(k, n);
    std::sort(order.begin(), order.begin() + keep);
    int32_t* out = idx + r * k;
    for (long long i = 0; i < k; ++i) out[i] = i < keep ? (int32_t)order[i] : -1;
  });
}

// [DSA-32K] Sparse Flash Attention forward, per token and head over the
// selected keys: s_i = scale q . kv[idx_i]; m = max s_i; l = sum exp(s_i - m);
// O = sum_i exp(s_i - m) / l * kv[idx_i, :d_v].  A token without a valid index
// gets O = 0, m = -inf, l = 0.
void dsa_ref_sparse_attn_fwd(long long B, long long S_q, long long S_k, long long H, long long d_qk,
                             long long d_v, long long k, const double* q, const double* kv,
                             const int32_t* idx, double scale, double* O, double* m, double* l,
                             int threads) {
  for_rows(B * S_q, threads, [&](long long r) {
    const long long b = r / S_q;
    const std::vector<long long> sel = selected(idx + r * k, k);
    const double* kvb = kv + b * S_k * d_qk;
    std::vector<double> s;
    for (long long h = 0; h < H; ++h) {
      double* Oh = O + (r * H + h) * d_v;
      for (long long e = 0; e < d_v; ++e) Oh[e] = 0.0;
      if (sel.empty()) {
        m[r * H + h] = kNegInf;
        l[r * H + h] = 0.0;
        continue;
      }
      logits(q + (r * H + h) * d_qk, kvb, d_qk, sel, scale, s);
      double mx = kNegInf;
      for (double x : s) mx = std::max(mx, x);
      double sum = 0.0;
      for (double x : s) sum += std::exp(x - mx);
      for (size_t i = 0; i < sel.size(); ++i) {
        const double p = std::exp(s[i] - mx) / sum;
        const double* v = kvb + sel[i] * d_qk;
        for (long long e = 0; e < d_v; ++e) Oh[e] += p * v[e];
      }
      m[r * H + h] = mx;
      l[r * H + h] = sum;
    }
  });
}

// [DSA-32K] SparseFlashAttentionGrad: P = exp(scale q.k - m) / l (recomputed
// from the saved statistics), D = sum_e dO * O, dP = dO V^T, dS = P (dP - D),
// dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO; dK (all d_qk columns) and
// dV (the first d_v) add into dkv.  dkv must be zeroed (or hold other rows'
// sums) by the caller.
void dsa_ref_sparse_attn_bwd(long long B, long long S_q, long long S_k, long long H,
                             long long d_qk, long long d_v, long long k, const double* q,
                             const double* kv, const int32_t* idx, const double* O,
                             const double* dO, const double* m, const double* l, double scale,
                             double* dq, double* dkv, int threads) {
  for_rows(B * S_q, threads, [&](long long r) {
    const long long b = r / S_q;
    const std::vector<long long> sel = selected(idx + r * k, k);
    const double* kvb = kv + b * S_k * d_qk;
    double* dkvb = dkv + b * S_k * d_qk;
    for (long long i = 0; i < H * d_qk; ++i) dq[r * H * d_qk + i] = 0.0;
    if (sel.empty()) return;
    const size_t n = sel.size();
    std::vector<double> dK(n * d_qk, 0.0), dV(n * d_v, 0.0), s;
    for (long long h = 0; h < H; ++h) {
      const double* qh = q + (r * H + h) * d_qk;
      const double* Oh = O + (r * H + h) * d_v;
      const double* dOh = dO + (r * H + h) * d_v;
      double* dqh = dq + (r * H + h) * d_qk;
      logits(qh, kvb, d_qk, sel, scale, s);
      double D = 0.0;
      for (long long e = 0; e < d_v; ++e) D += dOh[e] * Oh[e];
      for (size_t i = 0; i < n; ++i) {
        const double* kr = kvb + sel[i] * d_qk;
        const double P = std::exp(s[i] - m[r * H + h]) / l[r * H + h];
        double dP = 0.0;
        for (long long e = 0; e < d_v; ++e) dP += dOh[e] * kr[e];
        const double dS = P * (dP - D);
        for (long long d = 0; d < d_qk; ++d) {
          dqh[d] += scale * dS * kr[d];
          dK[i * d_qk + d] += scale * dS * qh[d];
        }
        for (long long e = 0; e < d_v; ++e) dV[i * d_v + e] += P * dOh[e];
      }
    }
    for (size_t i = 0; i < n; ++i) {
      double* row = dkvb + sel[i] * d_qk;
      for (long long d = 0; d < d_qk; ++d) atomic_add(row + d, dK[i * d_qk + d]);
      for (long long e = 0; e < d_v; ++e) atomic_add(row + e, dV[i * d_v + e]);
    }
  });
}

// [DSA-32K] SparseLightningIndexerGradKLLoss: target p = the attention
// probabilities (from m, l) summed over heads, L1-normalised over the
// selected keys; pi = Softmax(I) over the same keys with
// I_i = sum_j w_j ReLU(S_ji), S_ji = q_I[j] . k_I[idx_i]; loss_t = sum p log(p / pi);
// dI = pi - p; dw_j = sum_i dI_i ReLU(S_ji); dS_ji = dI_i w_j [S_ji > 0];
// dq_I[j] = sum_i dS_ji k_I[idx_i]; dk_I[idx_i] += sum_j dS_ji q_I[j].
// loss_rows [B*S_q] gets each token's loss; dk_I is accumulated.
void dsa_ref_indexer_kl_loss(long long B, long long S_q, long long S_k, long long H,
                             long long d_qk, long long H_I, long long d_I, long long k,
                             const double* q, const double* kv, const int32_t* idx,
                             const double* m, const double* l, double scale, const double* q_I,
                             const double* k_I, const double* w, double* loss_rows, double* dq_I,
                             double* dk_I, double* dw, int threads) {
  for_rows(B * S_q, threads, [&](long long r) {
    const long long b = r / S_q;
    const std::vector<long long> sel = selected(idx + r * k, k);
    const double* kvb = kv + b * S_k * d_qk;
    const double* kIb = k_I + b * S_k * d_I;
    for (long long i = 0; i < H_I * d_I; ++i) dq_I[r * H_I * d_I + i] = 0.0;
    for (long long j = 0; j < H_I; ++j) dw[r * H_I + j] = 0.0;
    loss_rows[r] = 0.0;
    if (sel.empty()) return;
    const size_t n = sel.size();
    // target: head sum of the attention probabilities, then L1 normalisation
    std::vector<double> p(n, 0.0), s;
    for (long long h = 0; h < H; ++h) {
      logits(q + (r * H + h) * d_qk, kvb, d_qk, sel, scale, s);
      for (size_t i = 0; i < n; ++i) p[i] += std::exp(s[i] - m[r * H + h]) / l[r * H + h];
    }
    double psum = 0.0;
    for (double x : p) psum += x;
    for (double& x : p) x /= psum;
    // indexer logits over the selected keys and their softmax
    std::vector<double> S(H_I * n), I(n, 0.0);
    for (long long j = 0; j < H_I; ++j) {
      const double* qj = q_I + (r * H_I + j) * d_I;
      for (size_t i = 0; i < n; ++i) {
        const double* ki = kIb + sel[i] * d_I;
        double dot = 0.0;
        for (long long d = 0; d < d_I; ++d) dot += qj[d] * ki[d];
        S[j * n + i] = dot;
        I[i] += w[r * H_I + j] * (dot > 0.0 ? dot : 0.0);
      }
    }
    double Imax = kNegInf;
    for (double x : I) Imax = std::max(Imax, x);
    double z = 0.0;
    for (double x : I) z += std::exp(x - Imax);
    const double lz = std::log(z);
    double loss = 0.0;
    std::vector<double> dI(n);
    for (size_t i = 0; i < n; ++i) {
      const double logpi = I[i] - Imax - lz;
      if (p[i] > 0.0) loss += p[i] * (std::log(p[i]) - logpi);
      dI[i] = std::exp(logpi) - p[i];
    }
    loss_rows[r] = loss;
    for (long long j = 0; j < H_I; ++j) {
      const double wj = w[r * H_I + j];
      const double* qj = q_I + (r * H_I + j) * d_I;
      double* dqj = dq_I + (r * H_I + j) * d_I;
      for (size_t i = 0; i < n; ++i) {
        const double Sji = S[j * n + i];
        dw[r * H_I + j] += dI[i] * (Sji > 0.0 ? Sji : 0.0);
        if (!(Sji > 0.0)) continue;
        const double dS = dI[i] * wj;
        const double* ki = kIb + sel[i] * d_I;
        double* dki = dk_I + (b * S_k + sel[i]) * d_I;
        for (long long d = 0; d < d_I; ++d) {
          dqj[d] += dS * ki[d];
          atomic_add(dki + d, dS * qj[d]);
        }
      }
    }
  });
}

int dsa_ref_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n > 0 ? (int)n : 1;
}

}  // extern "C"
