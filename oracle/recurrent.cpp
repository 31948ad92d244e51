// Oracle: token-by-token gated delta rule, forward and adjoint backward, in fp64.
//
// TEST INFRASTRUCTURE ONLY. This file is the checker for the CUDA library: only the
// tests, the smoke check and the benchmark's CPU-baseline leg may load it. It shares no
// code, header, table or helper with the CUDA path.
//
// What it computes (the plain definition the chunked algorithm reaches up to rounding):
// the gated delta rule recurrence as stated for Gated DeltaNet and its per-channel-gate
// variant (Kimi Delta Attention). The chunked eager reference on the hyper-parallel
// "Diff Coverage" page (function `torch_chunk_gated_delta_rule`, with its `_l2norm`
// helper) reaches this recurrence exactly up to rounding: its chunk loop carries the
// state S (K x V), decays it by exp(g), subtracts the prediction S^T k and writes back the
// beta-weighted innovation; the per-chunk output is q^T S read after the write.
//
// For one sequence (a dense batch row, or one document of a packed row) and one head,
// starting from S = S0 (or zeros):
//   qh = q * rsqrt(sum(q*q) + 1e-6),  kh likewise      (if use_l2norm; else qh=q, kh=k)
//   b  = sigmoid(beta) if use_beta_sigmoid else beta
//   S' = alpha (.) S   with alpha = exp(g_t) (scalar gate) or diag(exp(g_{t,k})) on rows k
//   delta = b * (v_t - S'^T kh)
//   S = S' + kh delta^T
//   o_t = scale * S^T qh
// The backward is the manual adjoint of those steps, run in reverse; states are
// checkpointed every 64 tokens and recomputed inside each block.
//
// Layout (all arrays fp64, row-major): q,k [R,H,K]; v [R,H,V]; g [R,H] (scalar gate) or
// [R,H,K] (per-channel); beta [R,H]; states [N,H,K,V]; o [R,H,V]. A sequence n covers rows
// [starts[n], starts[n]+lens[n]) of the flattened R = B*T rows.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

struct Problem {
  int n_seq, H, K, V;
  const int64_t* starts;
  const int64_t* lens;
  int per_channel;      // 1: gate is [R,H,K]
  int use_l2norm;
  int use_beta_sigmoid;
  double scale;
  const double *q, *k, *v, *g, *beta, *h0;  // h0 may be null
};

inline double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }

// Row-normalise x (length n) into y; return r = 1/sqrt(sum x^2 + eps).
inline double l2n(const double* x, double* y, int n) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += x[i] * x[i];
  double r = 1.0 / std::sqrt(s + 1e-6);
  for (int i = 0; i < n; ++i) y[i] = x[i] * r;
  return r;
}

struct TokenView {
  const double *q, *k, *v, *g;
  double beta;
};

inline TokenView token(const Problem& P, int64_t row, int h) {
  TokenView t;
  t.q = P.q + (row * P.H + h) * P.K;
  t.k = P.k + (row * P.H + h) * P.K;
  t.v = P.v + (row * P.H + h) * P.V;
  t.g = P.per_channel ? P.g + (row * P.H + h) * P.K : P.g + (row * P.H + h);
  t.beta = P.beta[row * P.H + h];
  return t;
}

// One forward step on S (K x V, row-major). Fills qh, kh, alpha (K entries), the
// decayed state Sp (optional), delta (V) and b. Returns nothing; S is updated in place.
void step_fwd(const Problem& P, const TokenView& t, std::vector<double>& S,
              std::vector<double>& qh, std::vector<double>& kh, std::vector<double>& alpha,
              std::vector<double>* Sp, std::vector<double>& pred, std::vector<double>& delta,
              double& b, double& rq, double& rk) {
  const int K = P.K, V = P.V;
  if (P.use_l2norm) {
    rq = l2n(t.q, qh.data(), K);
    rk = l2n(t.k, kh.data(), K);
  } else {
    rq = rk = 1.0;
    std::copy(t.q, t.q + K, qh.begin());
    std::copy(t.k, t.k + K, kh.begin());
  }
  b = P.use_beta_sigmoid ? sigmoid(t.beta) : t.beta;
  for (int i = 0; i < K; ++i) alpha[i] = std::exp(P.per_channel ? t.g[i] : t.g[0]);
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j) S[i * V + j] *= alpha[i];
  if (Sp) *Sp = S;
  for (int j = 0; j < V; ++j) {
    double s = 0.0;
    for (int i = 0; i < K; ++i) s += S[i * V + j] * kh[i];
    pred[j] = s;
    delta[j] = b * (t.v[j] - s);
  }
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j) S[i * V + j] += kh[i] * delta[j];
}

void run_fwd_chain(const Problem& P, int n, int h, double* o, double* hT) {
  const int K = P.K, V = P.V;
  std::vector<double> S(size_t(K) * V, 0.0), qh(K), kh(K), alpha(K), pred(V), delta(V);
  if (P.h0) {
    const double* s0 = P.h0 + (size_t(n) * P.H + h) * K * V;
    std::copy(s0, s0 + size_t(K) * V, S.begin());
  }
  for (int64_t tt = 0; tt < P.lens[n]; ++tt) {
    int64_t row = P.starts[n] + tt;
    TokenView t = token(P, row, h);
    double b, rq, rk;
    step_fwd(P, t, S, qh, kh, alpha, nullptr, pred, delta, b, rq, rk);
    double* out = o + (row * P.H + h) * V;
    for (int j = 0; j < V; ++j) {
      double s = 0.0;
      for (int i = 0; i < K; ++i) s += S[i * V + j] * qh[i];
      out[j] = P.scale * s;
    }
  }
  if (hT) {
    double* dst = hT + (size_t(n) * P.H + h) * K * V;
    std::copy(S.begin(), S.end(), dst);
  }
}

struct Grads {
  const double* dO;    // [R,H,V]
  const double* dhT;   // [N,H,K,V] or null
  double *dq, *dk, *dv, *dbeta, *dg, *dh0;  // dh0 may be null
};

void run_bwd_chain(const Problem& P, const Grads& G, int n, int h) {
  const int K = P.K, V = P.V;
  const int64_t len = P.lens[n], start = P.starts[n];
  const int blk = 64;
  const int64_t nblk = (len + blk - 1) / blk;
  // Forward pass storing the state entering every block of 64 tokens.
  std::vector<std::vector<double>> ckpt(static_cast<size_t>(nblk) + 1);
  std::vector<double> S(size_t(K) * V, 0.0), qh(K), kh(K), alpha(K), pred(V), delta(V);
  if (P.h0) {
    const double* s0 = P.h0 + (size_t(n) * P.H + h) * K * V;
    std::copy(s0, s0 + size_t(K) * V, S.begin());
  }
  for (int64_t bI = 0; bI < nblk; ++bI) {
    ckpt[bI] = S;
    for (int64_t tt = bI * blk; tt < std::min(len, (bI + 1) * blk); ++tt) {
      double b, rq, rk;
      step_fwd(P, token(P, start + tt, h), S, qh, kh, alpha, nullptr, pred, delta, b, rq, rk);
    }
  }
  // Reverse pass.
  std::vector<double> dS(size_t(K) * V, 0.0);
  if (G.dhT) {
    const double* s = G.dhT + (size_t(n) * P.H + h) * K * V;
    std::copy(s, s + size_t(K) * V, dS.begin());
  }
  std::vector<double> dqh(K), dkh(K), ddelta(V), dpred(V), Sp(size_t(K) * V);
  for (int64_t bI = nblk - 1; bI >= 0; --bI) {
    const int64_t t0 = bI * blk, t1 = std::min(len, (bI + 1) * blk);
    const int64_t nb = t1 - t0;
    // Recompute the states after each token of the block.
    const size_t nbs = static_cast<size_t>(nb);
    std::vector<std::vector<double>> Safter(nbs), Sdec(nbs);
    std::vector<std::vector<double>> QH(nbs), KH(nbs), AL(nbs), DL(nbs), PR(nbs);
    std::vector<double> Bv(nbs), RQ(nbs), RK(nbs);
    S = ckpt[bI];
    for (int64_t j = 0; j < nb; ++j) {
      double b, rq, rk;
      step_fwd(P, token(P, start + t0 + j, h), S, qh, kh, alpha, &Sp, pred, delta, b, rq, rk);
      Safter[j] = S; Sdec[j] = Sp; QH[j] = qh; KH[j] = kh; AL[j] = alpha; DL[j] = delta; PR[j] = pred;
      Bv[j] = b; RQ[j] = rq; RK[j] = rk;
    }
    for (int64_t j = nb - 1; j >= 0; --j) {
      const int64_t row = start + t0 + j;
      TokenView t = token(P, row, h);
      const double* dO = G.dO + (row * P.H + h) * V;
      const std::vector<double>& Sa = Safter[j];
      const std::vector<double>& Sd = Sdec[j];
      // o = scale * S^T qh
      for (int i = 0; i < K; ++i) {
        double s = 0.0;
        for (int c = 0; c < V; ++c) {
          dS[i * V + c] += P.scale * QH[j][i] * dO[c];
          s += Sa[i * V + c] * dO[c];
        }
        dqh[i] = P.scale * s;
      }
      // S = Sd + kh delta^T
      for (int c = 0; c < V; ++c) {
        double s = 0.0;
        for (int i = 0; i < K; ++i) s += dS[i * V + c] * KH[j][i];
        ddelta[c] = s;
      }
      for (int i = 0; i < K; ++i) {
        double s = 0.0;
        for (int c = 0; c < V; ++c) s += dS[i * V + c] * DL[j][c];
        dkh[i] = s;
      }
      // delta = b (v - pred)
      double db = 0.0;
      double* dv = G.dv + (row * P.H + h) * V;
      for (int c = 0; c < V; ++c) {
        dv[c] = Bv[j] * ddelta[c];
        db += ddelta[c] * (t.v[c] - PR[j][c]);
        dpred[c] = -Bv[j] * ddelta[c];
      }
      // pred = Sd^T kh
      for (int i = 0; i < K; ++i) {
        double s = 0.0;
        for (int c = 0; c < V; ++c) {
          dS[i * V + c] += KH[j][i] * dpred[c];
          s += Sd[i * V + c] * dpred[c];
        }
        dkh[i] += s;
      }
      // Sd = alpha (.) S_prev ; d(log alpha) = sum Sd (.) dS
      double* dg = P.per_channel ? G.dg + (row * P.H + h) * K : G.dg + (row * P.H + h);
      if (P.per_channel) {
        for (int i = 0; i < K; ++i) {
          double s = 0.0;
          for (int c = 0; c < V; ++c) s += Sd[i * V + c] * dS[i * V + c];
          dg[i] = s;
        }
      } else {
        double s = 0.0;
        for (size_t e = 0; e < dS.size(); ++e) s += Sd[e] * dS[e];
        dg[0] = s;
      }
      for (int i = 0; i < K; ++i)
        for (int c = 0; c < V; ++c) dS[i * V + c] *= AL[j][i];
      // beta transform
      double dbeta = db;
      if (P.use_beta_sigmoid) dbeta = db * Bv[j] * (1.0 - Bv[j]);
      G.dbeta[row * P.H + h] = dbeta;
      // l2 norm backward: dx = r (dxh - xh (xh . dxh))
      double* dq = G.dq + (row * P.H + h) * K;
      double* dk = G.dk + (row * P.H + h) * K;
      if (P.use_l2norm) {
        double sq = 0.0, sk = 0.0;
        for (int i = 0; i < K; ++i) { sq += QH[j][i] * dqh[i]; sk += KH[j][i] * dkh[i]; }
        for (int i = 0; i < K; ++i) {
          dq[i] = RQ[j] * (dqh[i] - QH[j][i] * sq);
          dk[i] = RK[j] * (dkh[i] - KH[j][i] * sk);
        }
      } else {
        for (int i = 0; i < K; ++i) { dq[i] = dqh[i]; dk[i] = dkh[i]; }
      }
    }
  }
  if (G.dh0) {
    double* dst = G.dh0 + (size_t(n) * P.H + h) * K * V;
    std::copy(dS.begin(), dS.end(), dst);
  }
}

template <class F>
void parallel_chains(const Problem& P, int threads, F f) {
  const int total = P.n_seq * P.H;
  if (threads <= 0) threads = int(std::thread::hardware_concurrency());
  threads = std::max(1, std::min(threads, total));
  std::vector<std::thread> pool;
  for (int w = 0; w < threads; ++w) {
    pool.emplace_back([&, w]() {
      for (int idx = w; idx < total; idx += threads) f(idx / P.H, idx % P.H);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Forward. o [R,H,V] is written for every row covered by a sequence; hT may be null.
// Returns 0 on success, -1 on bad arguments.
int oracle_gdr_fwd(int n_seq, const int64_t* starts, const int64_t* lens, int H, int K, int V,
                   int per_channel, int use_l2norm, int use_beta_sigmoid, double scale,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* beta, const double* h0, double* o, double* hT, int threads) {
  if (n_seq < 0 || H <= 0 || K <= 0 || V <= 0 || !starts || !lens) return -1;
  Problem P{n_seq, H, K, V, starts, lens, per_channel, use_l2norm, use_beta_sigmoid, scale,
            q, k, v, g, beta, h0};
  parallel_chains(P, threads, [&](int n, int h) { run_fwd_chain(P, n, h, o, hT); });
  return 0;
}

// Backward: gradients of sum(dO . o) + sum(dhT . hT) w.r.t. q, k, v, g (raw, per token),
// beta (as passed: the logit when use_beta_sigmoid) and h0.
int oracle_gdr_bwd(int n_seq, const int64_t* starts, const int64_t* lens, int H, int K, int V,
                   int per_channel, int use_l2norm, int use_beta_sigmoid, double scale,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* beta, const double* h0, const double* dO, const double* dhT,
                   double* dq, double* dk, double* dv, double* dbeta, double* dg, double* dh0,
                   int threads) {
  if (n_seq < 0 || H <= 0 || K <= 0 || V <= 0 || !starts || !lens) return -1;
  Problem P{n_seq, H, K, V, starts, lens, per_channel, use_l2norm, use_beta_sigmoid, scale,
            q, k, v, g, beta, h0};
  Grads G{dO, dhT, dq, dk, dv, dbeta, dg, dh0};
  parallel_chains(P, threads, [&](int n, int h) { run_bwd_chain(P, G, n, h); });
  return 0;
}

}  // extern "C"
