// tgdn_oracle.cpp — TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU statement of what rollback-free tree verification
// through Gated DeltaNet layers computes.  Only the tests, the smoke check and
// the benchmark's CPU-baseline leg may load it; the library never does.  It
// shares no code, header or constant table with the CUDA path.
//
// Source: "Trees from Marginals: Autoregressive drafting with factorized
// priors" (gist.science explainer pages, Technisches Resümee, Methodik 3,
// "Rollback-freie Baumverifizierung für GDN"):
//   * GDN update eq.:  S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T,
//     state d_k x d_v; the output of a token is o_t = S_t^T q_t.
//   * the tree is sorted topologically; per-branch verification walks every
//     branch with this recurrence ("pro-Zweig rekurrente Baselines",
//     Experimentelle Ergebnisse).  The oracle IS that walk: each node's state
//     is rebuilt from the committed state S0 along its own root path, sharing
//     nothing between branches, with no solve and no chunking.
//   * the state of the accepted node is committed once the accepted branch is
//     known (Methodik 3, last bullet); here that is the replayed state at the
//     accepted node.
//   * greedy acceptance: the longest root path whose draft tokens all agree
//     with the verifier's tokens (mean acceptance length, Experimentelle
//     Ergebnisse).
//
// Readings where the pages are silent (each also listed in the design notes):
//   * the root is a real token with its own q/k/v/g/b; its parent state is S0;
//   * g is the log-gate (a = exp(g)); q, k are used as given (no scaling);
//   * topological order = stable sort by (depth, index);
//   * v-head h reads query/key head h / (H_v / H_qk);
//   * acceptance ties (same depth) go to the smaller topological position.
//
// Build: g++ -O2 -std=c++17 -shared -fPIC -pthread (oracle/build.py).

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// Per-sequence tree status; the numbering is the library's documented
// contract, restated here.
enum {
  ST_OK = 0,
  ST_TOO_BIG = 1,     // more nodes than n_max
  ST_BAD_PARENT = 2,  // parent < -1, >= N, or the node itself
  ST_ROOTS = 3,       // not exactly one root
  ST_CYCLE = 4,       // some node never reaches the root
  ST_TOO_DEEP = 5,    // depth above depth_max
};

// Checks one sequence and computes the depth of every node by walking parents.
int check_tree(int N, const int32_t* par, int n_max, int depth_max, std::vector<int>& depth) {
  depth.assign(N, -1);
  if (N > n_max) return ST_TOO_BIG;
  for (int i = 0; i < N; ++i)
    if (par[i] < -1 || par[i] >= N || par[i] == i) return ST_BAD_PARENT;
  int roots = 0;
  for (int i = 0; i < N; ++i) roots += (par[i] == -1);
  if (N > 0 && roots != 1) return ST_ROOTS;
  for (int i = 0; i < N; ++i) {
    int j = i, hops = 0;
    while (par[j] != -1 && hops <= N) { j = par[j]; ++hops; }
    if (par[j] != -1) return ST_CYCLE;
    depth[i] = hops;
  }
  for (int i = 0; i < N; ++i)
    if (depth[i] > depth_max) return ST_TOO_DEEP;
  return ST_OK;
}

// Root path of node n, root first.
std::vector<int> root_path(const int32_t* par, int n) {
  std::vector<int> p;
  for (int j = n; j != -1; j = par[j]) p.push_back(j);
  return std::vector<int>(p.rbegin(), p.rend());
}

template <class F>
int parallel_for(long count, int nthreads, F&& body) {
  if (nthreads <= 0) nthreads = (int)std::thread::hardware_concurrency();
  if (nthreads < 1) nthreads = 1;
  if (nthreads > count) nthreads = (int)(count > 0 ? count : 1);
  std::atomic<long> next(0);
  auto worker = [&]() {
    for (long i = next++; i < count; i = next++) body(i);
  };
  std::vector<std::thread> pool;
  for (int t = 1; t < nthreads; ++t) pool.emplace_back(worker);
  worker();
  for (auto& t : pool) t.join();
  return nthreads;
}

struct Dims {
  int B, H_qk, H_v, dk, dv;
};

// One GDN step (the update eq.) on a d_k x d_v state, in place:
//   S <- a (S - b k (k^T S)) + b k v^T,  a = exp(g).
void gdn_step(std::vector<double>& S, int dk, int dv, const double* k, const double* v, double g,
              double b) {
  const double a = std::exp(g);
  std::vector<double> kS(dv, 0.0);  // k^T S
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) kS[j] += k[i] * S[(size_t)i * dv + j];
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) {
      double& s = S[(size_t)i * dv + j];
      s = a * (s - b * k[i] * kS[j]) + b * k[i] * v[j];
    }
}

// State of node n (local index) of sequence bi, v-head h, by replaying its root path.
void replay_state(const Dims& d, const int32_t* cu, const int32_t* par, const double* k,
                  const double* v, const double* g, const double* b, const double* S0, int bi,
                  int h, int n, std::vector<double>& S) {
  const int qh = h / (d.H_v / d.H_qk);
  const size_t ss = (size_t)d.dk * d.dv;
  S.assign(S0 + ((size_t)bi * d.H_v + h) * ss, S0 + ((size_t)bi * d.H_v + h + 1) * ss);
  for (int s : root_path(par + cu[bi], n)) {
    const size_t row = (size_t)cu[bi] + s;
    gdn_step(S, d.dk, d.dv, k + (row * d.H_qk + qh) * d.dk, v + (row * d.H_v + h) * d.dv,
             g[row * d.H_v + h], b[row * d.H_v + h]);
  }
}

}  // namespace

extern "C" {

// Tree metadata: depth, topological order (stable by depth, then index), its
// inverse pos, and the ancestor-or-self bitmask of every node, indexed by
// topological position: bit pos[s] of row pos[n] is set for each s on the
// root path of n, n included.  Invalid sequences get depth/order/pos = -1 and
// zero masks.  Returns 0, or -1 on a malformed batch description.
int oracle_prep(int B, const int32_t* cu, const int32_t* parent, int n_max, int depth_max,
                int words, int32_t* depth, int32_t* order, int32_t* pos, uint64_t* anc,
                int32_t* status) {
  if (B < 0 || words * 64 < n_max) return -1;
  std::vector<int> dep;
  for (int bi = 0; bi < B; ++bi) {
    const int lo = cu[bi], N = cu[bi + 1] - cu[bi];
    const int32_t* par = parent + lo;
    const int st = check_tree(N, par, n_max, depth_max, dep);
    status[bi] = st;
    for (int i = 0; i < N; ++i) {
      depth[lo + i] = order[lo + i] = pos[lo + i] = -1;
      for (int w = 0; w < words; ++w) anc[(size_t)(lo + i) * words + w] = 0;
    }
    if (st != ST_OK) continue;
    // stable order by depth: scan depths 0, 1, 2, ... and take nodes by index
    int p = 0;
    for (int dd = 0; p < N; ++dd)
      for (int i = 0; i < N; ++i)
        if (dep[i] == dd) order[lo + p++] = i;
    for (int q = 0; q < N; ++q) pos[lo + order[lo + q]] = q;
    for (int i = 0; i < N; ++i) {
      depth[lo + i] = dep[i];
      uint64_t* row = anc + (size_t)(lo + pos[lo + i]) * words;
      for (int s : root_path(par, i)) {
        const int ps = pos[lo + s];
        row[ps / 64] |= (uint64_t)1 << (ps % 64);
      }
    }
  }
  return 0;
}

// Greedy acceptance by brute force over all root paths.  A node is accepted
// when every non-root node on its root path (itself included) has
// target == draft; the root always is.  The accepted node is the deepest one,
// ties going to the smaller topological position.  path[bi] lists the root
// path root first, padded with -1 to depth_max + 1 entries.
int oracle_accept(int B, const int32_t* cu, const int32_t* parent, int n_max, int depth_max,
                  const int32_t* draft, const int32_t* target, int32_t* accept_node,
                  int32_t* accept_len, int32_t* path) {
  std::vector<int> dep;
  for (int bi = 0; bi < B; ++bi) {
    const int lo = cu[bi], N = cu[bi + 1] - cu[bi];
    const int32_t* par = parent + lo;
    accept_node[bi] = -1;
    accept_len[bi] = 0;
    for (int j = 0; j <= depth_max; ++j) path[(size_t)bi * (depth_max + 1) + j] = -1;
    if (check_tree(N, par, n_max, depth_max, dep) != ST_OK || N == 0) continue;
    int best = -1;
    for (int n = 0; n < N; ++n) {
      bool ok = true;
      for (int s : root_path(par, n))
        if (par[s] != -1 && target[lo + s] != draft[lo + s]) ok = false;
      if (!ok) continue;
      // stable (depth, index) order: deeper wins, then the smaller index
      if (best < 0 || dep[n] > dep[best]) best = n;
    }
    accept_node[bi] = best;
    accept_len[bi] = dep[best] + 1;
    const std::vector<int> rp = root_path(par, best);
    for (size_t j = 0; j < rp.size(); ++j) path[(size_t)bi * (depth_max + 1) + j] = rp[j];
  }
  return 0;
}

// Per-node outputs by path replay: o[row][h] = S_n^T q_n where S_n is the
// state after the root path of n.  Invalid sequences get zero outputs.
// Returns the number of threads used.
int oracle_verify(int B, const int32_t* cu, const int32_t* parent, int n_max, int depth_max,
                  int H_qk, int H_v, int dk, int dv, const double* q, const double* k,
                  const double* v, const double* g, const double* b, const double* S0, double* o,
                  int nthreads) {
  const Dims d{B, H_qk, H_v, dk, dv};
  return parallel_for((long)B * H_v, nthreads, [&](long item) {
    const int bi = (int)(item / H_v), h = (int)(item % H_v);
    const int lo = cu[bi], N = cu[bi + 1] - cu[bi];
    const int qh = h / (H_v / H_qk);
    std::vector<int> dep;
    const bool ok = check_tree(N, parent + lo, n_max, depth_max, dep) == ST_OK;
    std::vector<double> S;
    for (int n = 0; n < N; ++n) {
      double* out = o + ((size_t)(lo + n) * H_v + h) * dv;
      std::fill(out, out + dv, 0.0);
      if (!ok) continue;
      replay_state(d, cu, parent, k, v, g, b, S0, bi, h, n, S);
      const double* qn = q + ((size_t)(lo + n) * H_qk + qh) * dk;
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) out[j] += qn[i] * S[(size_t)i * dv + j];
    }
  });
}

// Committed state: the replayed state at accept_node[bi] (a local index).  A
// sequence with accept_node < 0 or an invalid tree keeps S0.  Returns the
// number of threads used.
int oracle_commit(int B, const int32_t* cu, const int32_t* parent, int n_max, int depth_max,
                  int H_qk, int H_v, int dk, int dv, const double* k, const double* v,
                  const double* g, const double* b, const double* S0,
                  const int32_t* accept_node, double* S_out, int nthreads) {
  const Dims d{B, H_qk, H_v, dk, dv};
  const size_t ss = (size_t)dk * dv;
  return parallel_for((long)B * H_v, nthreads, [&](long item) {
    const int bi = (int)(item / H_v), h = (int)(item % H_v);
    const int lo = cu[bi], N = cu[bi + 1] - cu[bi];
    double* out = S_out + ((size_t)bi * H_v + h) * ss;
    const double* s0 = S0 + ((size_t)bi * H_v + h) * ss;
    std::vector<int> dep;
    const int n = accept_node[bi];
    if (n < 0 || n >= N || check_tree(N, parent + lo, n_max, depth_max, dep) != ST_OK) {
      std::memcpy(out, s0, ss * sizeof(double));
      return;
    }
    std::vector<double> S;
    replay_state(d, cu, parent, k, v, g, b, S0, bi, h, n, S);
    std::memcpy(out, S.data(), ss * sizeof(double));
  });
}

}  // extern "C"
