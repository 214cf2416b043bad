// verify_tc.cu — tensor-core tree verification (bf16 io, d_k = d_v = 128, sm_103a).
//
// Single-pass verification of a draft tree through one GDN layer, following
// "Trees from Marginals" (Technisches Resümee, Methodik 3 and Implementierung:
// Gram matrix, forward substitution and output phase in one kernel).  With G
// the path-cumulative log-gate and A(n) / A*(n) the strict / inclusive
// ancestors of n,
//   X_ns = b_n e^{G_n-G_s} k_n.k_s  (s in A(n)),  Y_ns = e^{G_n-G_s} q_n.k_s  (s in A*(n))
//   (I + X) U = R = diag(b) (V - diag(e^G) K S0),   O = diag(e^G) Q S0 + Y U.
// Because X only links a node to its own ancestors, T = (I + X)^{-1} and
// W = Y T keep that sparsity, and row n of either depends only on the root
// path of n: it solves a (depth+1)-sized unit triangular system.  So
// U = T R and O = diag(e^G) Q S0 + W R, both tensor-core products.
//
// Persistent, warp-specialised kernel: one CTA per SM, 16 warps, looping over
// work items (sequence, v-head) that cover all 128 value columns (a contiguous
// run per CTA with a pending commit, else dealt round robin); trees have at most
// 64 nodes and depth at most 30.  Two items are in flight per SM:
//   producer warps 0-7, item j+1:
//     the item's fp32 state [128][128] arrives by one 64 KiB bulk copy over the
//     [K;Q] and state-operand areas; each thread takes one value column, 64 key
//     rows, into registers;
//     with a commit pending, the commit's product D^T = (C U_p)^T K_p runs on the
//     tensor cores (128 value columns x 64 key rows, twice, into the TMEM
//     columns the halves leave free) and each thread forms S = e^{G*} S + D;
//     S -> bf16 operand (K-major, 128-byte swizzle); TMA of the item's key and
//     query rows -> A = [K; Q]; tree metadata (staged in shared memory by
//     asynchronous copies an item ahead) ->
//     root paths (reused for the next head of the same sequence) and
//     path-cumulative gates; the committed state goes back to HBM last (warps
//     2-7 while warps 0-1 build the paths, once the metadata copies are out);
//   the producer's thread 255, item j+1, while the others build the metadata:
//     the first product into TMEM half (j+1) & 1,
//        D[:, 0:128] = A S0,  D[:, 128:192] = A K^T,
//     and, once it has read A and the operand, the bulk copy of the next item's
//     state into those areas;
//   consumer warps 8-15, item j:
//     Gram rows -> shared memory; V rows arrive by TMA and the key-lane warps
//     form R = diag(b)(V - e^G K S0) (bf16 hi/lo operand), clearing K S0 in
//     TMEM, while the query-lane warps substitute along the root paths, one T
//     or W row per thread with the partial sums in registers, writing straight
//     into the [T; W] operand;
//     tcgen05.mma accumulates [T; W'] R onto D[:, 0:128]: the key lanes end
//     with U = T R, the query lanes with Q S0 + W' R, W' = e^{-max(G,-60)} W,
//     so that O = e^{max(G,-60)} D;
//     U (workspace, fp32) and O (bf16) leave through swizzled shared-memory
//     staging and TMA tensor stores.
// The halves hand over through mbarriers: "stage 1 done" (the first product's
// completion plus the producer's metadata) and "TMEM half free".  Every wait is
// bounded: past the limit the CTA marks its items' sequences TGDN_SEQ_TIMEOUT,
// waits (bounded) for its own copies and products, frees its tensor memory
// and returns.  The kernel is launched with programmatic stream serialization:
// its prologue may overlap the previous kernel's tail and no input is read
// before griddepcontrol.wait.
// In a launch above 64 nodes it takes only the sequences of at most 64 nodes
// (small_only): up to 2048 sequences each CTA lists them (a warp ballot over cu_nodes)
// and numbers its items over that list; beyond that it deals every item and passes over
// the larger sequences without touching them.
// The state enters the tensor-core products as bf16 (fp32 accumulation); it is
// read, updated and written back in fp32.
//
// Deferred commit folded into the next verify (Methodik 3, last bullet: the
// state is committed once the accepted branch is known, in the following
// decode iteration).  When the previous step left a commit pending, the
// producer stages that step's accepted path for the item (u_s rows, k_s rows
// and G_s by 16-byte asynchronous copies, one item ahead, into an area of
// their own) and forms
//   S = e^{G*} S_prev + sum_{s on the path} e^{G*-G_s} k_s u_s^T
// with the sum as one tensor-core product, writes it back in place (the
// committed state) and verifies from it.  The state then crosses HBM once in
// each direction per step.
#include <type_traits>

#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kTcThreads = 512;
constexpr int kGroup = 256;    // threads per warp group (producer / consumer)
constexpr int kBarP = 1, kBarC = 2;  // hardware barrier ids of the two groups
constexpr int kBarM = 3;             // producer warps 0-1 (node metadata and root paths)
constexpr int kMetaThreads = 64;     // one node per thread
constexpr int kBarW = 4;             // all producer threads: paths done, state write-back
constexpr int kTcNodes = 64;   // nodes per tree on this kernel
constexpr int kTcDK = 128;
constexpr int kTcDV = 128;
constexpr int kTcDepth = 30;   // depth bound on this kernel
constexpr int kTcPath = kTcDepth + 1;  // entries of a root path
constexpr int kPathBytes = 32;         // one root path: a byte per depth, zero past the node
constexpr uint32_t kTmemCols = 512;    // two halves of 256 columns
constexpr int kGramCol = 128;          // within a half: [K;Q] S0 (0-127), Gram rows (128-191)
// The 64 columns each half leaves free hold the pending commit's product D^T: value
// column in the lane, key rows 0-63 at column 192 and rows 64-127 at column 448.
constexpr uint32_t kCommitCol0 = 192, kCommitCol1 = 448;

// Shared-memory map (bytes from a 1024-byte aligned base).
constexpr int kOffA = 0;          // [K;Q] operand: [2 d_k halves][128 rows][128 B]      32 KiB
// Before an item's [K;Q] rows and operand arrive, its fp32 state [128][128] (64 KiB)
// sits over both areas: one bulk copy, issued once the previous item's first product
// has read them.
constexpr int kOffState = 0;
constexpr int kOffS = 32768;      // S0^T operand (bf16), K-major [2 k halves][128 columns][128 B]
// While the pending commit is formed the same area holds its operands (path padded to
// 32 entries): (C U_p)^T hi and lo, MN-major [2 m chunks][4 k groups][8][128 B], and
// K_p, MN-major [2 n chunks][4 k groups][8][128 B].
constexpr int kOffCAhi = kOffS;
constexpr int kOffCAlo = kOffS + 8192;
constexpr int kOffCB = kOffS + 16384;
// Pending-commit staging, an area of its own so that the next item's rows are in
// flight while this item's operands are still being read:
constexpr int kOffUP = 65536;                         // u_s rows [kTcPath][128] fp32   15.5 KiB
constexpr int kOffKP = kOffUP + kTcPath * kTcDV * 4;  // k_s rows [kTcPath][128] bf16   7.75 KiB
constexpr int kOffGP = kOffKP + kTcPath * kTcDK * 2;  // 16-byte chunks holding G_s [kTcPath]
// Gram rows: K K^T rows [64][kKKStride] fp32 (padded: a column read by lanes that share
// a row, or a row read at distinct columns, hits distinct banks), then Q K^T rows
// [64][64] fp32 with the 16-byte chunks of row n rotated by n & 7.
constexpr int kKKStride = 68;
constexpr int kOffKK = 90112;
constexpr int kOffQK = kOffKK + 64 * kKKStride * 4;
constexpr int kOffRhi = 131072;   // R operand, MN-major [2 col atoms][8 node groups][8][128 B]
constexpr int kOffRlo = 147456;
constexpr int kOffA2hi = 163840;  // [T; W] operand, K-major [16 row groups][8][128 B]     16 KiB
constexpr int kOffA2lo = 180224;
static_assert(kOffGP + kTcPath * 16 <= kOffKK, "commit staging fits its area");
static_assert(kOffQK + 64 * 64 * 4 <= kOffRhi, "Gram rows fit their area");
// Small values the producer needs an item later arrive by 4- and 8-byte asynchronous
// copies into two parity slots, so that no register carries them across an iteration
// and nothing waits on them before the item's first barrier: the node metadata of the
// next item (and the ancestor mask of each topological position), and the pending
// commit's accepted path two items ahead (lane l: entry l) with that sequence's bounds.
struct NodeStage {
  int dep[kTcNodes], pos[kTcNodes], ord[kTcNodes];
  float gg[kTcNodes], bb[kTcNodes];
  uint64_t anc[kTcNodes];
};
struct CommitStage {
  int path[32];
  int lo, hi, st, pad;
};
constexpr int kOffNS = kOffQK + 64 * 64 * 4;  // the gap after the Gram rows
constexpr int kOffCS = kOffNS + 2 * (int)sizeof(NodeStage);
static_assert(kOffNS % 16 == 0 && kOffCS % 16 == 0 &&
                  kOffCS + 2 * (int)sizeof(CommitStage) <= kOffRhi,
              "metadata staging fits between the Gram rows and the R operand");
constexpr int kOffMeta = 196608;
constexpr int kMaxCompact = 2048;  // sequences of a mixed launch that can be listed
// Output staging after the second product, in the 128-byte swizzled tile layout of
// the TMA stores that send it out: U in the Gram-row area (free once the solve is
// done), O in an area of its own after the shared state (below), so that the next
// item only waits for the U tiles to be read before it stores its Gram rows.
constexpr int kOffUst = kOffKK;     // U: 4 tiles (32 columns each) [64 rows][128 B] fp32
static_assert(kOffUst % 1024 == 0 && kOffUst + 4 * 8192 <= kOffRhi,
              "U staging: 1024-byte aligned tiles in the Gram-row area");

struct alignas(16) ItemMeta {
  uint8_t path[kTcNodes][kPathBytes];  // [node][depth]: the node's ancestor at that depth
  int lo, N, h, good;
  int skip;   // a sequence above 64 nodes in a mixed launch: nothing to do here
  int zrows;  // rows zero-filled when the item is not verified
  int dep[kTcNodes];
  int ord[kTcNodes];
  int pos[kTcNodes];
  float gg[kTcNodes];
  float G[kTcNodes];
  float bb[kTcNodes];
};
struct TcShared {
  uint64_t tma_bar, mma1_bar, mma2_bar, v_bar;
  uint64_t s1_done[2];    // consumer waits: first product done + metadata written
  uint64_t cmt_bar;       // producer waits: the commit product is in TMEM
  uint64_t st_bar;        // producer waits: an item's state has landed
  uint64_t tmem_free[2];  // producer waits: consumer finished the item in this half
  uint32_t tmem_slot;
  int abort;
  int tma_issued;
  int v_issued;
  int mma1_issued;
  int mma2_issued;
  int cmt_issued;
  int st_issued;
  int c_L[2];             // staged path length per item parity (0: nothing to commit)
  int c_row[2][kTcPath];  // previous-step node rows of the staged path
  int c_gi[2][kTcPath];   // index of G_s within its staged 16-byte chunk
  ItemMeta meta[2];
  // Mixed launches: the sequences of at most 64 nodes in order (items are numbered
  // over them, so that the CTAs only get items of this kernel).
  int n_small;
  int16_t small_seq[kMaxCompact];
};
// O: 2 tiles (64 columns each) [64 rows][128 B] bf16, 1024-byte aligned
constexpr int kOffOst = (kOffMeta + (int)sizeof(TcShared) + 1023) / 1024 * 1024;
constexpr int kTcSmemBytes = kOffOst + 2 * 8192 + 1024;  // + alignment slack
static_assert(kTcSmemBytes <= 227 * 1024, "fits one CTA per SM");

// 16-byte chunk swizzle of the 128-byte-row operands (TMA and tcgen05
// SWIZZLE_128B layout for 1024-byte aligned 8-row atoms).
__device__ __forceinline__ int swz(int row, int chunk) { return chunk ^ (row & 7); }
__device__ __forceinline__ int atom_off(int row, int chunk) {
  return (row >> 3) * 1024 + (row & 7) * 128 + (swz(row, chunk) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// x ~= hi + lo with hi = bf16(x), lo = bf16(x - hi), for 8 consecutive values.
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  float h[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = __bfloat162float(__float2bfloat16_rn(x[i]));
  hi = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]),
                  pack_bf16x2(h[6], h[7]));
  lo = make_uint4(pack_bf16x2(x[0] - h[0], x[1] - h[1]), pack_bf16x2(x[2] - h[2], x[3] - h[3]),
                  pack_bf16x2(x[4] - h[4], x[5] - h[5]), pack_bf16x2(x[6] - h[6], x[7] - h[7]));
}

// One thread of a warp group waits on the mbarrier (suspending, bounded); the
// rest of the group parks on the group's hardware barrier, which also makes
// the outcome the same for every thread of the group.
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, int bar_id,
                                           bool leader, volatile int* abort, uint64_t limit_ns) {
  bool ok = true;
  if (leader) ok = mbar_wait_suspend(bar, parity, abort, limit_ns);
  return named_sync_and(bar_id, kGroup, ok);
}

// The same over a named barrier of n threads.
__device__ __forceinline__ bool group_wait_n(uint64_t* bar, uint32_t parity, int bar_id, int n,
                                             bool leader, volatile int* abort, uint64_t limit_ns) {
  bool ok = true;
  if (leader) ok = mbar_wait_suspend(bar, parity, abort, limit_ns);
  return named_sync_and(bar_id, n, ok);
}

// The bounds and status of the next item's sequence (its node metadata is staged in
// shared memory).
struct Prefetch {
  int lo, N, st;
};

// v[k] for a run-time k in [0, N), N a power of two: a binary multiplexer over
// the bits of k (fixed register indices, log2 N dependent selects).
template <int N>
__device__ __forceinline__ float pick(const float (&v)[N], int k) {
  float t[N];
#pragma unroll
  for (int m = 0; m < N; ++m) t[m] = v[m];
#pragma unroll
  for (int w = N / 2, bit = 0; w >= 1; w /= 2, ++bit) {
    const bool hi = (k >> bit) & 1;
#pragma unroll
    for (int m = 0; m < w; ++m) t[m] = hi ? t[2 * m + 1] : t[2 * m];
  }
  return t[0];
}

// v[k] for k in [LO, LO + R) (R a power of two, the range within v): the same
// multiplexer over R candidates only.  (k outside the range picks some candidate.)
template <int LO, int R, int N>
__device__ __forceinline__ float pick_range(const float (&v)[N], int k) {
  static_assert(LO >= 0 && LO + R <= N && (R & (R - 1)) == 0, "range within the sums");
  const int d = k - LO;
  float t[R];
#pragma unroll
  for (int m = 0; m < R; ++m) t[m] = v[LO + m];
#pragma unroll
  for (int w = R / 2, bit = 0; w >= 1; w /= 2, ++bit) {
    const bool hi = (d >> bit) & 1;
#pragma unroll
    for (int m = 0; m < w; ++m) t[m] = hi ? t[2 * m + 1] : t[2 * m];
  }
  return t[0];
}

// Byte j of the packed root path (a node index).
__device__ __forceinline__ int path_at(const uint32_t (&pw)[8], int j) {
  return static_cast<int>((pw[j >> 2] >> (8 * (j & 3))) & 0xffu);
}

// acc[j] += s * row[p_j] for j < W (row: a shared-memory address).  Only j < i - 1
// matter at step i; the other entries are either the next one (taken out before) or
// settled ones, never read again, so the width only has to cover i - 1 (no per-entry
// test).  The W loads are issued back to back before the first multiply-add, so
// their latencies overlap.
template <int W, int N>
__device__ __forceinline__ void path_update(float (&acc)[N], const uint32_t (&pw)[8], float s,
                                            uint32_t row) {
  static_assert(W <= N, "width within the partial sums");
  float v[W];
#pragma unroll
  for (int j = 0; j < W; ++j)
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[j]) : "r"(row + 4u * path_at(pw, j)));
#pragma unroll
  for (int j = 0; j < W; ++j) acc[j] = fmaf(s, v[j], acc[j]);
}

// One row of T (t_row) or W of the node sn at depth dn, by substitution along
// its root path P = (p_0 = root, ..., p_dn = sn):
//   r (I + X_P) = y,  X_P[i][j] = b_{p_i} e^{G_{p_i} - G_{p_j}} k_{p_i}.k_{p_j} (i > j),
//   y = e_dn for T;  y_j = e^{G_n - G_{p_j}} q_n.k_{p_j} for W.
// The gates leave the recurrence once each entry is rescaled to
// rho_j = r_j e^{G_{p_j} - G_n}:
//   rho_j = y'_j - acc_j,  acc_j = sum_{i>j} b_{p_i} rho_i k_{p_i}.k_{p_j},
//   y' = e_dn for T;  y'_j = q_n.k_{p_j} for W,
// and r_j = rho_j e^{G_n - G_{p_j}} (at most 1 for non-positive gates) is only
// formed for the store, off the chain of dependent operations.
// Entries are settled from the node towards the root; once s_i = b_{p_i} rho_i
// is known it is added into every acc_j (j < i) at once.  acc lives in
// registers; the loop runs from the warp's deepest row, so the step index i is
// the same in every lane.  The next entry's sum is taken out of acc before the
// update and only its own term is added, so the chain from one entry to the
// next is a subtract, a multiply and a fused multiply-add; the Gram reads and
// the other updates are off it.  r_j is written as bf16 hi + lo at column p_j
// of the [T; W] operand row.
template <int D>
__device__ __forceinline__ void solve_path_row(const ItemMeta& M, const float* KK,
                                               const float* QK, uint8_t* smem, int sn, int dn,
                                               int wmax, bool t_row) {
  constexpr int NA = D <= 16 ? 16 : 32;  // partial sums held (entries 0 .. NA-1)
  static_assert(D <= NA, "path fits the partial sums");
  const uint8_t* prow = M.path[sn];  // entries past the node are 0 (a valid node)
  const uint4* pr = reinterpret_cast<const uint4*>(prow);
  const uint4 pa = pr[0], pb = pr[1];
  const uint32_t pw[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
  const float Gn = M.G[sn];
  const int a2row = t_row ? sn : 64 + sn;
  // a W row is stored times e^{-max(G_n, -60)}: the second product adds it onto
  // Q S0 and the output is that sum times e^{max(G_n, -60)}
  const float gofs = t_row ? Gn : Gn - fmaxf(Gn, -60.f);
  const float* GRq = QK + sn * 64;  // q_n . k_s (chunks rotated by sn & 7)
  const int xq = (sn & 7) << 2;
  float acc[NA];
#pragma unroll
  for (int k = 0; k < NA; ++k) acc[k] = 0.f;
  float ai = 0.f;  // acc_i of the current step
  // Software pipeline: the path entry two steps ahead and the gate, beta and
  // query-Gram value one step ahead are loaded before they are needed.
  int pi = prow[wmax];
  int pn = wmax > 0 ? prow[wmax - 1] : 0;  // the next entry's node
  float Gi = M.G[pi], bi = M.bb[pi];
  float qi = t_row ? 0.f : GRq[pi ^ xq];
  // One step at index i: its update width W (entries 0 .. W-1 cover 0 .. i-2) and the
  // range [LO, LO + R) that holds acc_{i-1}.
  auto step = [&](int i, auto Wc, auto LOc, auto Rc) {
    constexpr int W = decltype(Wc)::value, LO = decltype(LOc)::value, R = decltype(Rc)::value;
    const int pnn = i > 1 ? prow[i - 2] : 0;
    const float Gnx = M.G[pn], bnx = M.bb[pn];
    const float qnx = t_row ? 0.f : GRq[pn ^ xq];
    const float* GRi = KK + pi * kKKStride;  // K K^T row p_i (padded, unrotated)
    const uint32_t GRs = smem_addr(GRi);
    const float kn = GRi[pn];                // k_{p_i}.k_{p_{i-1}}
    const float yp = t_row ? (i == dn ? 1.f : 0.f) : qi;
    const float base = pick_range<LO, R>(acc, i - 1);  // acc_{i-1} before this step's term
    const float rho = yp - ai;
    const bool own = i <= dn;
    const float s = own ? rho * bi : 0.f;
    if (own) {
      const float rw = rho * __expf(gofs - Gi);
      const __nv_bfloat16 hi = __float2bfloat16_rn(rw);
      const __nv_bfloat16 lw = __float2bfloat16_rn(rw - __bfloat162float(hi));
      const int off = atom_off(a2row, pi >> 3) + (pi & 7) * 2;
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2hi + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2lo + off) = lw;
    }
    path_update<W>(acc, pw, s, GRs);
    ai = fmaf(s, kn, base);
    pi = pn;
    pn = pnn;
    Gi = Gnx;
    bi = bnx;
    qi = qnx;
  };
  using C4 = std::integral_constant<int, 4>;
  using C8 = std::integral_constant<int, 8>;
  using C12 = std::integral_constant<int, 12>;
  using C16 = std::integral_constant<int, 16>;
  if constexpr (NA == 16) {
    // Four phases by the width of the update (i - 1 in [13, 15], [9, 12], [5, 8],
    // [-1, 4]); within a phase acc_{i-1} is one of 4 (or 8) entries, a small
    // multiplexer instead of one over all 16.  (At i = 0 the picked value is unused.)
    int i = wmax;
    for (; i >= 14; --i) step(i, C16{}, std::integral_constant<int, 12>{}, C4{});
    for (; i >= 10; --i) step(i, C12{}, std::integral_constant<int, 9>{}, C4{});
    for (; i >= 6; --i) step(i, C8{}, std::integral_constant<int, 5>{}, C4{});
    for (; i >= 0; --i) step(i, C4{}, std::integral_constant<int, 0>{}, C8{});
  } else {
    for (int i = wmax; i >= 0; --i) {
      const int pnn = i > 1 ? prow[i - 2] : 0;
      const float Gnx = M.G[pn], bnx = M.bb[pn];
      const float qnx = t_row ? 0.f : GRq[pn ^ xq];
      const float* GRi = KK + pi * kKKStride;  // K K^T row p_i (padded, unrotated)
      const uint32_t GRs = smem_addr(GRi);
      const float kn = GRi[pn];                // k_{p_i}.k_{p_{i-1}}
      const float yp = t_row ? (i == dn ? 1.f : 0.f) : qi;
      const float base = pick<NA>(acc, i - 1);  // acc_{i-1} before this step's term
      const float rho = yp - ai;
      const bool own = i <= dn;
      const float s = own ? rho * bi : 0.f;
      if (own) {
        const float rw = rho * __expf(gofs - Gi);
        const __nv_bfloat16 hi = __float2bfloat16_rn(rw);
        const __nv_bfloat16 lw = __float2bfloat16_rn(rw - __bfloat162float(hi));
        const int off = atom_off(a2row, pi >> 3) + (pi & 7) * 2;
        *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2hi + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(smem + kOffA2lo + off) = lw;
      }
      const int lim = i - 1;  // entries 0 .. i-2 take their terms here
      if (lim <= 4) {
        path_update<4>(acc, pw, s, GRs);
      } else if (lim <= 8) {
        path_update<8>(acc, pw, s, GRs);
      } else if (lim <= 12) {
        path_update<12>(acc, pw, s, GRs);
      } else if (lim <= 16) {
        path_update<16>(acc, pw, s, GRs);
      } else if (lim <= 24) {
        path_update<(NA < 24 ? NA : 24)>(acc, pw, s, GRs);
      } else {
        path_update<NA>(acc, pw, s, GRs);
      }
      ai = fmaf(s, kn, base);
      pi = pn;
      pn = pnn;
      Gi = Gnx;
      bi = bnx;
      qi = qnx;
    }
  }
}

template <int kSolveD>
__global__ void __launch_bounds__(kTcThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap, const __grid_constant__ OutMaps om,
                 int n_items, int H_qk, int H_v, int depth_max, int words, int small_only,
                 int compact, const int32_t* __restrict__ cu,
                 const int32_t* __restrict__ depth, const int32_t* __restrict__ order,
                 const int32_t* __restrict__ pos, const uint64_t* __restrict__ anc,
                 int32_t* __restrict__ status,
                 const float* __restrict__ g, const float* __restrict__ bta, float* S,
                 __nv_bfloat16* __restrict__ o, float* __restrict__ Uws,
                 float* __restrict__ Gws, const PendingCommit cm, const uint64_t wait_ns,
                 const int hold_item) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcShared& sh = *reinterpret_cast<TcShared*>(smem + kOffMeta);
  volatile int* abort = &sh.abort;
  const int tid = threadIdx.x, warp = tid >> 5;
  if ((int)blockIdx.x >= n_items) return;
  // Item order.  With a pending commit the producer warps are the critical path,
  // so each CTA takes a contiguous run of items: consecutive items are mostly the
  // heads of one sequence, whose root paths are then reused.  Otherwise the items
  // are dealt round robin, so that the CTAs work on neighbouring heads of the
  // same rows at the same time (better DRAM locality for the v, U and o rows).
  const bool runs = cm.path != nullptr;
  int i_begin = runs ? (int)(((long)blockIdx.x * n_items) / gridDim.x) : (int)blockIdx.x;
  int i_end = runs ? (int)(((long)(blockIdx.x + 1) * n_items) / gridDim.x) : n_items;
  const int i_step = runs ? 1 : (int)gridDim.x;
  const int grp = H_v / H_qk;  // v-heads per query/key head
  const bool fused = cm.path != nullptr;
  // Launched with programmatic stream serialization: everything up to
  // griddepcontrol.wait below touches no global memory (the first item's state
  // is only pulled into L2, which stays coherent), so it can overlap the tail of
  // the previous kernel in the stream.
  if (tid == 0 && !compact) prefetch_l2(S + (size_t)i_begin * kTcDK * kTcDV, kTcDK * kTcDV * 4);

  if (tid == 0) {
    mbar_init(&sh.tma_bar, 1);
    mbar_init(&sh.mma1_bar, 1);
    mbar_init(&sh.mma2_bar, 1);
    mbar_init(&sh.v_bar, 1);
    mbar_init(&sh.s1_done[0], 2);
    mbar_init(&sh.s1_done[1], 2);
    mbar_init(&sh.cmt_bar, 1);
    mbar_init(&sh.st_bar, 1);
    mbar_init(&sh.tmem_free[0], 1);
    mbar_init(&sh.tmem_free[1], 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    sh.abort = 0;
    sh.tma_issued = 0;
    sh.v_issued = 0;
    sh.mma1_issued = 0;
    sh.mma2_issued = 0;
    sh.cmt_issued = 0;
    sh.st_issued = 0;
  }
  if (warp == 0) tmem_alloc(&sh.tmem_slot, kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_slot;
  grid_dependency_wait();     // the previous kernel's writes are visible from here on
  grid_launch_dependents();   // the next kernel may start its own prologue
  if (compact) {
    // A mixed launch lists its sequences of at most 64 nodes (warp 0, a ballot per 32
    // sequences) and numbers its items over them; a CTA left without items leaves.
    if (warp == 0) {
      const int B = n_items / H_v;
      const int lane = tid & 31;
      int base = 0;
      for (int b0 = 0; b0 < B; b0 += 32) {
        const int b = b0 + lane;
        const bool sm = b < B && cu[b + 1] - cu[b] <= kTcNodes;
        const unsigned m = __ballot_sync(0xffffffffu, sm);
        if (sm) sh.small_seq[base + __popc(m & ((1u << lane) - 1u))] = static_cast<int16_t>(b);
        base += __popc(m);
      }
      if (lane == 0) sh.n_small = base;
    }
    __syncthreads();
    const int ni = sh.n_small * H_v;
    i_begin = runs ? (int)(((long)blockIdx.x * ni) / gridDim.x) : (int)blockIdx.x;
    i_end = runs ? (int)(((long)(blockIdx.x + 1) * ni) / gridDim.x) : ni;
    if (i_begin >= i_end) {
      if (warp == 0) tmem_dealloc(tmem, kTmemCols);
      return;
    }
  } else if (small_only) {  // a CTA whose items all belong to the 128-node kernel leaves at once
    int mine = 0;
    if (warp == 0)
      for (int it = i_begin + (tid & 31) * i_step; it < i_end; it += 32 * i_step) {
        const int n = cu[it / H_v + 1] - cu[it / H_v];
        mine |= (n > 0 && n <= kTcNodes) ? 1 : 0;
      }
    if (!__syncthreads_or(mine)) {
      if (warp == 0) tmem_dealloc(tmem, kTmemCols);
      return;
    }
  }

  // the sequence of an item (listed in a mixed launch) and the offset of its state
  auto seq_of = [&](int it) { return compact ? (int)sh.small_seq[it / H_v] : it / H_v; };
  auto state_block = [&](int it) {
    return ((size_t)seq_of(it) * H_v + it % H_v) * (size_t)(kTcDK * kTcDV);
  };

  if (tid < kGroup) {
    // =================================================== producer warps 0-7
    const int p = tid;
    auto issue_kq = [&](int item, int row0) {  // thread 0 only; row0 = cu[item / H_v]
      const int qh = (item % H_v) / grp;
      mbar_arrive_expect_tx(&sh.tma_bar, 4 * 64 * 128);
      // box = 64 d_k elements x 1 head x 64 node rows, 128-byte swizzled rows
      tma_load_3d(smem + kOffA + 0, &kmap, &sh.tma_bar, 0, qh, row0);
      tma_load_3d(smem + kOffA + 8192, &qmap, &sh.tma_bar, 0, qh, row0);
      tma_load_3d(smem + kOffA + 16384, &kmap, &sh.tma_bar, 64, qh, row0);
      tma_load_3d(smem + kOffA + 24576, &qmap, &sh.tma_bar, 64, qh, row0);
      sh.tma_issued += 1;
    };
    // The state of one item, one value column per thread: warp w holds column
    // jc = 32 (w & 3) + lane of key rows rb .. rb + 63, rb = 64 (w >> 2), read from the
    // bulk copy in shared memory (with a pending commit the kernel writes these rows
    // back from registers).  A warp's access to one row is one 128-byte line, and the
    // registers line up with the TMEM lanes of the commit product (lane = value
    // column).
    const int jc = 32 * ((p >> 5) & 3) + (p & 31);
    const int rb = 64 * (p >> 7);
    float sreg[64];
    auto issue_state = [&](int item) {  // thread 0 only
      mbar_arrive_expect_tx(&sh.st_bar, kTcDK * kTcDV * 4);
      bulk_load(smem + kOffState, S + state_block(item), kTcDK * kTcDV * 4,
                &sh.st_bar);
      sh.st_issued += 1;
    };
    NodeStage* const NS = reinterpret_cast<NodeStage*>(smem + kOffNS);
    CommitStage* const CS = reinterpret_cast<CommitStage*>(smem + kOffCS);
    // Warp 0, two items ahead of its staging: the item's accepted path in the
    // previous tree (lane l copies entry l) and that sequence's bounds and status,
    // into parity slot x.  (Raw values: they are combined when the item is
    // published, an iteration later, after this thread's cp_async_wait_all.)
    auto load_commit_meta = [&](int it, int x) {
      const int bi = seq_of(it);
      CommitStage& cs = CS[x];
      cp_async4(&cs.path[p],
                cm.path + (size_t)bi * cm.path_len + (p < cm.path_len ? p : cm.path_len - 1));
      if (p == 0) {
        cp_async4(&cs.lo, cm.cu + bi);
        cp_async4(&cs.hi, cm.cu + bi + 1);
        cp_async4(&cs.st, cm.status + bi);
      }
    };
    // Warp 0: the item's staged path (entries after the first invalid one are
    // ignored) -> c_L[cb], c_row[cb].
    auto publish_commit = [&](int cb) {
      __syncwarp();  // lane 0's copies (the bounds) are visible to the whole warp
      const CommitStage& cs = CS[cb];
      const int c_plo = cs.lo, c_phi = cs.hi, c_st = cs.st, c_node = cs.path[p];
      const bool valid = c_st == TGDN_SEQ_OK && p < cm.path_len && c_node >= 0 &&
                         c_node < c_phi - c_plo;
      const int L = __ffs(__ballot_sync(0xffffffffu, !valid)) - 1;  // path_len <= 31
      if (p == 0) sh.c_L[cb] = L;
      if (p < L) sh.c_row[cb][p] = c_plo + c_node;
    };
    // All producer threads: 16-byte asynchronous copies of the published path's
    // u_s rows, k_s rows and the chunks holding G_s (49 chunks per path node).
    auto stage_commit = [&](int it, int cb) {
      const int h = it % H_v, qh = h / grp;
      const int L = sh.c_L[cb];
      for (int e = p; e < L * 49; e += kGroup) {
        const int l = e / 49, w = e - l * 49;
        const size_t row = static_cast<size_t>(sh.c_row[cb][l]);
        if (w < 32) {
          cp_async16(smem + kOffUP + l * (kTcDV * 4) + w * 16,
                     cm.U + (row * H_v + h) * kTcDV + w * 4);
        } else if (w < 48) {
          cp_async16(smem + kOffKP + l * (kTcDK * 2) + (w - 32) * 16,
                     static_cast<const __nv_bfloat16*>(cm.k) + (row * H_qk + qh) * kTcDK +
                         (w - 32) * 8);
        } else {
          const size_t ge = row * H_v + h;  // the workspace base is 256-byte aligned
          sh.c_gi[cb][l] = static_cast<int>(ge & 3);
          cp_async16(smem + kOffGP + l * 16, cm.G + (ge & ~static_cast<size_t>(3)));
        }
      }
      cp_async_commit();
    };
    // Sequence bounds and status one item ahead of the node metadata, so that no
    // load waits on another load of the same iteration (raw bounds: the count is
    // formed when they are used).
    int q_lo = 0, q_hi = 0, q_st = 0;
    auto load_seq = [&](int item) {
      const int bi = seq_of(item);
      q_lo = cu[bi];
      q_hi = cu[bi + 1];
      q_st = status[bi];
    };
    Prefetch pf;
    // The bounds come from load_seq; warps 0-1 copy the node metadata (node p) and the
    // ancestor mask of topological position p (word 0: positions < 64) into slot x.
    auto load_meta = [&](int item, int x) {
      pf.lo = q_lo;
      pf.N = q_hi - q_lo;
      pf.st = q_st;
      // (rows of a sequence whose bounds tree prep found bad are never touched)
      if (p < kMetaThreads && pf.st == TGDN_SEQ_OK && p < pf.N) {
        const size_t r = (size_t)(pf.lo + p);
        const int h = item % H_v;
        NodeStage& ns = NS[x];
        cp_async4(&ns.dep[p], depth + r);
        cp_async4(&ns.pos[p], pos + r);
        cp_async4(&ns.ord[p], order + r);
        cp_async4(&ns.gg[p], g + r * H_v + h);
        cp_async4(&ns.bb[p], bta + r * H_v + h);
        cp_async8(&ns.anc[p], anc + r * words);
      }
    };
    int item = i_begin;
    // (the first item's commit path does not depend on its bounds: it goes out first,
    // as a copy group of its own, so that its staging need not wait for them)
    if (fused && p < 32) {
      load_commit_meta(item, 0);
      cp_async_commit();
    }
    load_seq(item);
    load_meta(item, 0);
    cp_async_commit();
    if (item + i_step < i_end) load_seq(item + i_step);
    if (p == 0 && !(small_only && pf.N > kTcNodes)) issue_state(item);
    if (fused) {
      if (p < 32) {
        cp_async_wait_all_but_last();  // the commit path (the metadata may still be in flight)
        publish_commit(0);
      }
      named_sync(kBarP, kGroup);
      stage_commit(item, 0);
      if (p < 32 && item + i_step < i_end) load_commit_meta(item + i_step, 1);
    }

    int prev_bi = -1;  // sequence of the previous item when its tree was valid
    int npr = 0;       // items processed so far (passed-over items excluded): one [K;Q]
                       // copy and one first product each, in order
    int ncm = 0;       // commit products issued so far
    int nst = 0;       // state copies consumed so far
    for (int j = 0; item < i_end; ++j, item += i_step) {
      const int slot = j & 1;
      ItemMeta& M = sh.meta[slot];
      const int bi = seq_of(item), h = item % H_v;
      // this thread's column of the item's state (key rows rb .. rb + 63)
      float* const s_col = S + ((size_t)bi * H_v + h) * (size_t)(kTcDK * kTcDV) +
                           (size_t)rb * kTcDV + jc;
      const int lo = pf.lo, N = pf.N;
      const int next = item + i_step;
      // (small_only: sequences above 64 nodes belong to the 128-node kernel; their
      // items pass through without state, solve or writes)
      const bool skip = small_only && N > kTcNodes;
      bool ok = (pf.st == TGDN_SEQ_OK) && N > 0 && N <= kTcNodes;
      // this item's state, from the bulk copy into the [K;Q] and operand areas
      if (!skip) {
        if (!group_wait(&sh.st_bar, nst & 1, kBarP, p == 0, abort, wait_ns)) break;
        ++nst;
        const float* st = reinterpret_cast<const float*>(smem + kOffState) + rb * kTcDV + jc;
#pragma unroll
        for (int i = 0; i < 64; ++i) sreg[i] = st[i * kTcDV];
      }
      int L = 0;
      // this thread's staged copies (commit rows, node metadata, path words) have landed
      if (fused || p < kMetaThreads) cp_async_wait_all();
      if (fused && p < 32 && next < i_end) publish_commit(slot ^ 1);  // the next item's path
      // every thread has read its state rows (and the staged rows are visible to the
      // group after the barrier): the areas are free for this item's [K;Q] rows and the
      // commit operands
      fence_proxy_async_smem();
      if (!named_sync_and(kBarP, kGroup, !*abort)) break;
      if (fused) L = sh.c_L[slot];
      if (p == 0 && !skip) issue_kq(item, lo);
      if (L > 0) {
        // The previous step's commit, S = e^{G*} S + sum_l e^{G*-G_l} k_l u_l^T, on the
        // tensor cores: D^T = (C U_p)^T K_p with C = diag(e^{G*-G_l}) (M = 128 value
        // columns, N = 2 x 64 key rows, K = the path padded to 16 or 32; C U_p as bf16
        // hi + lo, K_p exact), then S = e^{G*} S + D in registers.
        const int kp = L <= 16 ? 16 : 32;
        const int kcs = kp / 8 * 1024;  // bytes per 64-element chunk of an operand
        const float* UP = reinterpret_cast<const float*>(smem + kOffUP);
        const uint4* KP = reinterpret_cast<const uint4*>(smem + kOffKP);
        const float* GP = reinterpret_cast<const float*>(smem + kOffGP);
        const float Gstar = GP[(L - 1) * 4 + sh.c_gi[slot][L - 1]];
        for (int u = p; u < kp * 16; u += kGroup) {
          const int l = u >> 4, mc = u & 15;  // path entry; 8-element chunk of its row
          const int off = (mc >> 3) * kcs + (l >> 3) * 1024 + (l & 7) * 128 +
                          (((mc & 7) ^ (l & 7)) << 4);
          uint4 ahi = make_uint4(0u, 0u, 0u, 0u), alo = ahi, bk = ahi;
          if (l < L) {
            const float cl = __expf(Gstar - GP[l * 4 + sh.c_gi[slot][l]]);
            const float4 u0 = reinterpret_cast<const float4*>(UP + l * kTcDV)[2 * mc];
            const float4 u1 = reinterpret_cast<const float4*>(UP + l * kTcDV)[2 * mc + 1];
            const float x[8] = {cl * u0.x, cl * u0.y, cl * u0.z, cl * u0.w,
                                cl * u1.x, cl * u1.y, cl * u1.z, cl * u1.w};
            split8(x, ahi, alo);
            bk = KP[l * (kTcDK / 8) + mc];
          }
          *reinterpret_cast<uint4*>(smem + kOffCAhi + off) = ahi;
          *reinterpret_cast<uint4*>(smem + kOffCAlo + off) = alo;
          *reinterpret_cast<uint4*>(smem + kOffCB + off) = bk;
        }
        fence_proxy_async_smem();
        named_sync(kBarP, kGroup);  // the commit operands are written
        if (p == 0) {
          tc_fence_after_sync();
          const uint32_t sAh = smem_addr(smem + kOffCAhi), sAl = smem_addr(smem + kOffCAlo);
          const uint32_t sB = smem_addr(smem + kOffCB);
          constexpr uint32_t id_c = idesc_bf16_f32(128, 64, 1, 1);
          for (int ks = 0; ks < kp / 16; ++ks) {
            // MN-major operands: 64-element chunks kcs apart, 8-entry k groups 1 KiB apart
            const uint64_t ah = smem_desc(sAh + ks * 2048, kcs, 1024, kSwizzle128B);
            const uint64_t al = smem_desc(sAl + ks * 2048, kcs, 1024, kSwizzle128B);
#pragma unroll
            for (int nh = 0; nh < 2; ++nh) {
              const uint64_t bd = smem_desc(sB + nh * kcs + ks * 2048, kcs, 1024, kSwizzle128B);
              const uint32_t d = tmem + (nh ? kCommitCol1 : kCommitCol0);
              umma_bf16(d, ah, bd, id_c, ks > 0);
              umma_bf16(d, al, bd, id_c, 1);
            }
          }
          umma_commit(&sh.cmt_bar);
          sh.cmt_issued += 1;
        }
        if (!group_wait(&sh.cmt_bar, ncm & 1, kBarP, p == 0, abort, wait_ns)) break;
        ++ncm;
        tc_fence_after_sync();
        const float decay = __expf(Gstar);
        const uint32_t tc0 = tmem + (static_cast<uint32_t>(32 * ((p >> 5) & 3)) << 16) +
                             (rb == 0 ? kCommitCol0 : kCommitCol1);
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
          float d[32];
          tmem_ld32(tc0 + hv * 32, d);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) sreg[hv * 32 + i] = fmaf(decay, sreg[hv * 32 + i], d[i]);
        }
      }
      // The bf16 copy of the (committed) state into the K-major operand; the state
      // itself goes back and the next item's comes in after this item is handed over
      // (the memory traffic then overlaps the consumer's work on this item).  (The
      // state enters the tensor-core product as bf16; it stays fp32 in memory.)
      if (!skip) {
        uint8_t* op_row = smem + kOffS + (rb >> 6) * 16384 + jc * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)  // 8 key rows per 16-byte chunk
          *reinterpret_cast<uint4*>(op_row + ((c8 ^ (jc & 7)) << 4)) =
              make_uint4(pack_bf16x2(sreg[c8 * 8], sreg[c8 * 8 + 1]),
                         pack_bf16x2(sreg[c8 * 8 + 2], sreg[c8 * 8 + 3]),
                         pack_bf16x2(sreg[c8 * 8 + 4], sreg[c8 * 8 + 5]),
                         pack_bf16x2(sreg[c8 * 8 + 6], sreg[c8 * 8 + 7]));
      }
      fence_proxy_async_smem();
      named_sync(kBarP, kGroup);  // the S operand is complete
      // From here the group splits three ways until warps 0-1 have their paths:
      // thread 255 issues the first product, warps 0-1 (one node per thread) build the
      // metadata and root paths, and warps 2-7 wait to send their committed state back.
      // A wait that gives up raises *abort; the group then leaves together at the
      // next item's first barrier (or the loop ends).
      //
      // Thread 255 (no node of its own) issues the first product into TMEM half `slot`
      // once the consumer has finished item j-2 (the previous user of the half) and
      // this item's key and query rows have landed,
      //   D[:, 0:128] = [K;Q] S0,  D[:, 128:192] = [K;Q] K^T,
      // and, once that product has read the [K;Q] and operand areas, copies the next
      // item's state there.  A passed-over item gets no product.  (A test hook can
      // withhold one item's product: the consumer's bounded wait for it then expires.)
      if (p == kGroup - 1) {
        bool ok255 = true;
        if (hold_item >= 0 && seq_of(item) * H_v + item % H_v == hold_item) {
          ok255 = false;
        } else if (skip) {
          mbar_arrive(&sh.s1_done[slot]);
        } else if ((ok255 = (j < 2 || mbar_wait_suspend(&sh.tmem_free[slot], ((j >> 1) + 1) & 1,
                                                         abort, wait_ns)) &&
                            mbar_wait_suspend(&sh.tma_bar, npr & 1, abort, wait_ns))) {
          tc_fence_after_sync();
          const uint32_t tb1 = tmem + slot * 256;
          const uint32_t sA = smem_addr(smem + kOffA);
          const uint32_t sS = smem_addr(smem + kOffS);
          constexpr uint32_t id_s0 = idesc_bf16_f32(128, 128, 0, 0);
          constexpr uint32_t id_gram = idesc_bf16_f32(128, kTcNodes, 0, 0);
#pragma unroll
          for (int s2 = 0; s2 < kTcDK / 16; ++s2) {
            const uint64_t ad = smem_desc(sA + (s2 >> 2) * 16384 + (s2 & 3) * 32, 16, 1024,
                                          kSwizzle128B);
            // K-major S0^T: the same layout as A (64-element k halves 16 KiB apart)
            const uint64_t hd = smem_desc(sS + (s2 >> 2) * 16384 + (s2 & 3) * 32, 16, 1024,
                                          kSwizzle128B);
            umma_bf16(tb1, ad, hd, id_s0, s2 > 0);
            umma_bf16(tb1 + kGramCol, ad, ad, id_gram, s2 > 0);  // B = the key rows of A
          }
          umma_commit(&sh.mma1_bar);
          umma_commit(&sh.s1_done[slot]);
          sh.mma1_issued += 1;
        }
        const int n1 = npr + (skip ? 0 : 1);  // first products issued so far
        if (ok255 && next < i_end && !(small_only && q_hi - q_lo > kTcNodes) &&
            (n1 == 0 || mbar_wait_suspend(&sh.mma1_bar, (n1 - 1) & 1, abort, wait_ns)))
          issue_state(next);
      }
      if (p < kMetaThreads) {
        // Warps 0-1: this slot's node metadata once the consumer is done with item j-2
        // (its previous user), then the root paths.
        bool go = j < 2 || group_wait_n(&sh.tmem_free[slot], ((j >> 1) + 1) & 1, kBarM,
                                        kMetaThreads, p == 0, abort, wait_ns);
        const NodeStage& ns = NS[slot];
        if (go) {
          if (p == 0) {
            M.lo = lo;
            M.N = N;
            M.h = h;
            M.skip = skip;
            // rows zero-filled for an item that is not verified: none for a passed-over
            // item or for a sequence whose bounds tree prep found bad
            M.zrows = (skip || pf.st == TGDN_SEQ_BAD_RANGE || N < 0) ? 0 : N;
          }
          if (ok && p < N) {
            const int dp = ns.dep[p], ps = ns.pos[p], od = ns.ord[p];
            if (dp >= 0 && dp <= depth_max && dp <= kTcDepth && ps >= 0 && ps < N && od >= 0 &&
                od < N) {
              M.dep[p] = dp;
              M.pos[p] = ps;
              M.ord[p] = od;
              M.gg[p] = ns.gg[p];
              M.bb[p] = ns.bb[p];
            } else {
              ok = false;
            }
          }
        }
        // the next item's metadata and a later item's commit bounds go out now (into
        // the other slots); they land while this item's paths are built
        if (next < i_end) load_meta(next, slot ^ 1);
        if (p < 32 && fused && next + i_step < i_end) load_commit_meta(next + i_step, slot);
        // those copies are out: warps 2-7 may now fill the global-memory path with the
        // commit staging and their share of the state write-back
        named_arrive(kBarW, kGroup);
        if (go) {
          named_sync(kBarM, kMetaThreads);  // this slot's node metadata is written
          // root paths from the ancestor masks (bits = topological positions,
          // ascending = root first) and path-cumulative log-gates; the same tree as
          // the previous item (another head) reuses its paths and only sums the gates.
          // A node index read from another thread's metadata is range-checked before
          // it is used (the group agrees on validity only after this).
          const bool reuse = prev_bi == bi;
          if (ok && p < N && reuse) {
            const int dn = M.dep[p];
            const uint8_t* srow_p = sh.meta[slot ^ 1].path[p];
            const uint4* src = reinterpret_cast<const uint4*>(srow_p);
            uint4* dst = reinterpret_cast<uint4*>(M.path[p]);
            dst[0] = src[0];
            dst[1] = src[1];
            float acc = 0.f;
            for (int i = 0; i <= dn; ++i) acc += M.gg[srow_p[i]];
            M.G[p] = acc;
          } else if (ok && p < N) {
            const int dn = M.dep[p];
            uint64_t mk = ns.anc[M.pos[p]];  // this node's ancestor mask (by its position)
            bool pk = __popcll(mk) == dn + 1 && ((mk >> M.pos[p]) & 1ull);
            uint8_t* prow = M.path[p];
            reinterpret_cast<uint4*>(prow)[0] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(prow)[1] = make_uint4(0u, 0u, 0u, 0u);
            float acc = 0.f;
            int last = -1;
            for (int i = 0; pk && i <= dn; ++i) {
              const int b = __ffsll(static_cast<long long>(mk)) - 1;
              mk &= mk - 1;
              if (b >= N) {
                pk = false;
                break;
              }
              const int s = M.ord[b];
              if (s < 0 || s >= N) {
                pk = false;
                break;
              }
              pk = M.dep[s] == i;
              prow[i] = static_cast<uint8_t>(s);
              acc += M.gg[s];
              last = s;
            }
            if (!pk || last != p) ok = false;
            M.G[p] = acc;
          }
          ok = named_sync_and(kBarM, kMetaThreads, ok);
          prev_bi = ok ? bi : -1;
          if (p == 0) {
            M.good = ok;
            mbar_arrive(&sh.s1_done[slot]);  // the metadata above is written
          }
        }
      }
      // Warps 2-7 stage the next commit and send their share of the state back once warps
      // 0-1 have issued their metadata copies (a burst of stores issued earlier would sit
      // in the global-memory path ahead of them: measured, the metadata phase then took
      // up to twice as long); warps 0-1 follow after their paths.
      if (p >= kMetaThreads) named_sync(kBarW, kGroup);
      // (every thread takes the next item's bounds and status, which decide whether
      // it is passed over; only warps 0-1 load node metadata)
      if (p >= kMetaThreads && next < i_end) load_meta(next, slot ^ 1);
      if (next < i_end && next + i_step < i_end) load_seq(next + i_step);
      if (fused && next < i_end) stage_commit(next, slot ^ 1);
      if (!skip) ++npr;
      // the committed state back in place (fused; L2-only stores: the state is touched
      // once per step and never by this SM again within the launch)
      if (L > 0) {
#pragma unroll
        for (int i = 0; i < 64; ++i) __stcg(s_col + (size_t)i * kTcDV, sreg[i]);
      }
      // A block boundary here keeps the compiler from moving the next iteration's work
      // in among these memory instructions (measured: that interleaving made the
      // launch ~7% slower; a plain memory clobber is not enough, a branch is).
      if (p == 0) asm volatile("" ::: "memory");
    }
  } else {
    // =================================================== consumer warps 8-15
    const int c = tid - kGroup;
    const int cw = c >> 5;            // 0..7
    const int lq = cw & 3;            // TMEM lane quarter (warp index mod 4)
    const int chalf = cw >> 2;        // value-column half
    const uint32_t lane_base = static_cast<uint32_t>(lq * 32) << 16;
    const int lane_row = lq * 32 + (c & 31);
    const bool key_lane = lq < 2;
    const int lane_node = key_lane ? lane_row : lane_row - 64;
    // Thread 0, one item ahead: the V rows of an item go by TMA into the R lo
    // operand area (the same swizzled layout), where R is then formed in place.
    int cv_lo = 0, cv_hi = 0;  // node rows of the item whose V rows go out next
    auto load_vseq = [&](int item) {
      cv_lo = cu[seq_of(item)];
      cv_hi = cu[seq_of(item) + 1];
    };
    // a passed-over item (small_only, above 64 nodes) gets no V rows
    auto v_wanted = [&]() { return !(small_only && cv_hi - cv_lo > kTcNodes); };
    auto issue_v = [&](int item) {
      mbar_arrive_expect_tx(&sh.v_bar, 2 * 64 * 128);
      tma_load_3d(smem + kOffRlo, &vmap, &sh.v_bar, 0, item % H_v, cv_lo);
      tma_load_3d(smem + kOffRlo + 8192, &vmap, &sh.v_bar, 64, item % H_v, cv_lo);
      sh.v_issued += 1;
    };
    int item = i_begin;
    if (c == 0) {
      load_vseq(item);
      if (v_wanted()) issue_v(item);
      if (item + i_step < i_end) load_vseq(item + i_step);
    }
    uint32_t mma2_count = 0;  // second products issued so far (same in every thread)
    int nv = 0;               // V copies consumed so far (one per item not passed over)
    for (int j = 0; item < i_end; ++j, item += i_step) {
      const int slot = j & 1;
      const int next = item + i_step;
      if (!group_wait(&sh.s1_done[slot], (j >> 1) & 1, kBarC, c == 0, abort, wait_ns)) break;
      tc_fence_after_sync();
      const ItemMeta& M = sh.meta[slot];
      const int lo = M.lo, N = M.N, h = M.h;
      const uint32_t tb = tmem + slot * 256;

      if (!M.good) {  // bad or empty sequence: zero rows (none for a passed-on item)
        const int nz = M.zrows;
        for (int e = c; e < nz * (kTcDV / 4); e += kGroup) {
          const int n = e >> 5, c4 = e & 31;
          const size_t row = ((size_t)(lo + n) * H_v + h) * kTcDV + c4 * 4;
          *reinterpret_cast<uint2*>(o + row) = make_uint2(0u, 0u);
          *reinterpret_cast<float4*>(Uws + row) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int n = c; n < nz; n += kGroup) Gws[(size_t)(lo + n) * H_v + h] = 0.f;
        bool v_ok = true;
        if (c == 0) {  // this item's V rows have landed: the area is free for the next
          if (!M.skip) v_ok = mbar_wait_suspend(&sh.v_bar, nv & 1, abort, wait_ns);
          if (v_ok && next < i_end) {
            if (v_wanted()) issue_v(next);
            if (next + i_step < i_end) load_vseq(next + i_step);
          }
        }
        if (!M.skip) ++nv;
        if (!named_sync_and(kBarC, kGroup, v_ok)) break;
        if (c == 0) mbar_arrive(&sh.tmem_free[slot]);
        continue;
      }

      // ---- Gram rows -> shared memory; [T; W] operand zeroed
      {
        float r[32];
        tmem_ld32(tb + lane_base + kGramCol + chalf * 32, r);
        tmem_ld_wait();
        // the previous item's U tiles (the older of its two store groups) have been
        // read out of the Gram-row area
        if (c == 0) bulk_wait_read_but_last();
        named_sync(kBarC, kGroup);
        if (key_lane) {  // K K^T row lane_row
          float4* dst = reinterpret_cast<float4*>(smem + kOffKK) +
                        (lane_row * kKKStride + chalf * 32) / 4;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            dst[c4] = make_float4(r[c4 * 4], r[c4 * 4 + 1], r[c4 * 4 + 2], r[c4 * 4 + 3]);
        } else {  // Q K^T row lane_node
          float* QK = reinterpret_cast<float*>(smem + kOffQK) + lane_node * 64;
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            *reinterpret_cast<float4*>(QK + swz(lane_node, chalf * 8 + c4) * 4) =
                make_float4(r[c4 * 4], r[c4 * 4 + 1], r[c4 * 4 + 2], r[c4 * 4 + 3]);
        }
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < 8; ++i)  // 32 KiB of [T; W] hi + lo, consecutive 16 B per thread
          *reinterpret_cast<uint4*>(smem + kOffA2hi + (i * kGroup + c) * 16) = zero;
      }
      named_sync(kBarC, kGroup);  // Gram rows stored, [T; W] operand zeroed

      // Key-lane warps form R while the query-lane warps solve for T and W (the
      // solve needs only the Gram rows and the metadata).
      // ---- R = diag(b)(V - e^G K S0) as a bf16 hi/lo operand (key lanes, a column
      // half per warp); the K S0 columns are zeroed once read: the second product
      // accumulates U = T R there
      bool v_ok = true;
      if (key_lane) {
        v_ok = mbar_wait_suspend(&sh.v_bar, nv & 1, abort, wait_ns);
        const bool live = lane_node < N;
        const float eG = live ? __expf(M.G[lane_node]) : 0.f;
        const float bn = live ? M.bb[lane_node] : 0.f;
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // 32 value columns at a time
          float r[32];
          tmem_ld32(tb + lane_base + chalf * 64 + q * 32, r);
          tmem_ld_wait();
          {
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
            tmem_st32(tb + lane_base + chalf * 64 + q * 32, z);
          }
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {  // 8 columns per 16-byte bf16 chunk
            const int off = chalf * 8192 + atom_off(lane_node, q * 4 + c8);
            const uint4 vv = *reinterpret_cast<const uint4*>(smem + kOffRlo + off);
            const __nv_bfloat162* vb = reinterpret_cast<const __nv_bfloat162*>(&vv);
            float xr[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 vf = __bfloat1622float2(vb[i]);
              xr[2 * i] = live ? bn * (vf.x - eG * r[c8 * 8 + 2 * i]) : 0.f;
              xr[2 * i + 1] = live ? bn * (vf.y - eG * r[c8 * 8 + 2 * i + 1]) : 0.f;
            }
            uint4 hi, lw;
            split8(xr, hi, lw);  // rows of R beyond the tree are exact zeros
            *reinterpret_cast<uint4*>(smem + kOffRhi + off) = hi;
            *reinterpret_cast<uint4*>(smem + kOffRlo + off) = lw;
          }
        }
        tmem_st_wait();
      } else {
        // ---- the rows of T (lane quarter 2) and of W (lane quarter 3), one row per
        // thread.  Rows are handed out in topological order: the column-half-0 warps
        // take the first 32 positions, the others the deeper 32, so each scheduler
        // runs one shallow and one deep solve.
        const float* KK = reinterpret_cast<const float*>(smem + kOffKK);
        const float* QK = reinterpret_cast<const float*>(smem + kOffQK);
        const bool t_row = lq == 2;
        const int spos = chalf * 32 + (c & 31);
        const bool act = spos < N;
        const int sn = act ? M.ord[spos] : 0;
        const int dn = act ? M.dep[sn] : -1;
        const int wmax = __reduce_max_sync(0xffffffffu, dn);
        solve_path_row<kSolveD>(M, KK, QK, smem, sn, dn, wmax, t_row);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      if (!named_sync_and(kBarC, kGroup, v_ok)) break;
      tc_fence_after_sync();

      // ---- second product, added onto columns 0-127: key lanes (zeroed) get U = T R,
      // query lanes Q S0 + W' R with W' = e^{-max(G, -60)} W  (hi.hi + hi.lo + lo.hi)
      if (c == 0) {
        const uint32_t sA2hi = smem_addr(smem + kOffA2hi);
        const uint32_t sA2lo = smem_addr(smem + kOffA2lo);
        const uint32_t sRhi = smem_addr(smem + kOffRhi);
        const uint32_t sRlo = smem_addr(smem + kOffRlo);
        constexpr uint32_t id_r = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
        for (int s = 0; s < kTcNodes / 16; ++s) {
          const uint64_t ah = smem_desc(sA2hi + s * 32, 16, 1024, kSwizzle128B);
          const uint64_t al = smem_desc(sA2lo + s * 32, 16, 1024, kSwizzle128B);
          // MN-major R: value-column atoms 8 KiB apart, 8-node groups 1 KiB apart
          const uint64_t bh = smem_desc(sRhi + s * 2048, 8192, 1024, kSwizzle128B);
          const uint64_t bl = smem_desc(sRlo + s * 2048, 8192, 1024, kSwizzle128B);
          umma_bf16(tb, ah, bh, id_r, 1);
          umma_bf16(tb, ah, bl, id_r, 1);
          umma_bf16(tb, al, bh, id_r, 1);
        }
        umma_commit(&sh.mma2_bar);
        sh.mma2_issued += 1;
      }
      if (c == 0) bulk_wait_read();  // the previous item's O tiles have left their staging
      const bool done2 = group_wait(&sh.mma2_bar, mma2_count & 1, kBarC, c == 0, abort, wait_ns);
      ++mma2_count;
      if (!done2) break;
      tc_fence_after_sync();
      // the operand areas are free: the next item's V rows go out now
      ++nv;
      if (c == 0 && next < i_end) {
        if (v_wanted()) issue_v(next);
        if (next + i_step < i_end) load_vseq(next + i_step);
      }

      // ---- key lanes: U rows; query lanes: O = e^G Q S0 + W R (bf16).  Rows are
      // staged in 128-byte swizzled tiles and leave by a few TMA tensor stores (a box
      // of 64 rows, else boxes of 8); the last N mod 8 rows, which a box of 8 would
      // overrun into the next sequence, go out from registers.
      {
        const bool live = lane_node < N;
        const bool direct = live && lane_node >= (N & ~7);
        const int sw = lane_node & 7;
        if (key_lane) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            float r[32];
            tmem_ld32(tb + lane_base + chalf * 64 + q * 32, r);
            tmem_ld_wait();
            uint8_t* row = smem + kOffUst + (chalf * 2 + q) * 8192 + lane_node * 128;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<float4*>(row + ((i ^ sw) << 4)) =
                  make_float4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
            if (direct) {
              float4* dst = reinterpret_cast<float4*>(
                  Uws + ((size_t)(lo + lane_node) * H_v + h) * kTcDV + chalf * 64 + q * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
            }
          }
          if (live && chalf == 0) Gws[(size_t)(lo + lane_node) * H_v + h] = M.G[lane_node];
        } else {
          uint8_t* row = smem + kOffOst + chalf * 8192 + lane_node * 128;
          uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(lo + lane_node) * H_v + h) * kTcDV +
                                                chalf * 64);
          // O = e^{max(G, -60)} (Q S0 + W' R); below e^{-60} the Q S0 term is far
          // under fp32 resolution of the W R term
          const float eG = live ? __expf(fmaxf(M.G[lane_node], -60.f)) : 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // 16 value columns at a time
            float a[16];
            tmem_ld16(tb + lane_base + chalf * 64 + q * 16, a);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float* aa = a + 8 * i;
              const uint4 pk = make_uint4(pack_bf16x2(eG * aa[0], eG * aa[1]),
                                          pack_bf16x2(eG * aa[2], eG * aa[3]),
                                          pack_bf16x2(eG * aa[4], eG * aa[5]),
                                          pack_bf16x2(eG * aa[6], eG * aa[7]));
              *reinterpret_cast<uint4*>(row + (((q * 2 + i) ^ sw) << 4)) = pk;
              if (direct) dst[q * 2 + i] = pk;
            }
          }
        }
      }
      fence_proxy_async_smem();  // the staged rows are visible to the tensor stores
      tc_fence_before_sync();
      named_sync(kBarC, kGroup);
      if (c == 0) {
        mbar_arrive(&sh.tmem_free[slot]);  // this half is free again
        const int n8 = N & ~7;
        // two store groups, U first: the next item waits only for the U tiles
        for (int r0 = 0; r0 < n8;) {
          const bool big = r0 == 0 && n8 == 64;
          const CUtensorMap* um = big ? &om.u64 : &om.u8;
#pragma unroll
          for (int t = 0; t < 4; ++t)
            tma_store_3d(um, smem + kOffUst + t * 8192 + r0 * 128, t * 32, h, lo + r0);
          r0 += big ? 64 : 8;
        }
        bulk_commit();
        for (int r0 = 0; r0 < n8;) {
          const bool big = r0 == 0 && n8 == 64;
          const CUtensorMap* omp = big ? &om.o64 : &om.o8;
#pragma unroll
          for (int t = 0; t < 2; ++t)
            tma_store_3d(omp, smem + kOffOst + t * 8192 + r0 * 128, t * 64, h, lo + r0);
          r0 += big ? 64 : 8;
        }
        bulk_commit();
      }
    }
    bulk_wait_all();  // this thread's output rows are written
  }

  // ---- end.  After an expired wait every item still owned by this CTA is
  // reported as timed out, and the latest copies and products are drained (bounded).
  cp_async_wait_all();  // staging copies left by a loop that ended early
  __syncthreads();
  if (sh.abort && tid == 0) {
    for (int it2 = i_begin; it2 < i_end; it2 += i_step)
      atomicCAS(&status[seq_of(it2)], TGDN_SEQ_OK, TGDN_SEQ_TIMEOUT);
    if (sh.tma_issued > 0) (void)mbar_wait(&sh.tma_bar, (sh.tma_issued - 1) & 1, wait_ns);
    if (sh.v_issued > 0) (void)mbar_wait(&sh.v_bar, (sh.v_issued - 1) & 1, wait_ns);
  }
  // the last products, before TMEM and the operands are released (bounded)
  if (tid == 0 && sh.mma1_issued > 0) (void)mbar_wait(&sh.mma1_bar, (sh.mma1_issued - 1) & 1, wait_ns);
  if (tid == 0 && sh.mma2_issued > 0) (void)mbar_wait(&sh.mma2_bar, (sh.mma2_issued - 1) & 1, wait_ns);
  if (tid == 0 && sh.cmt_issued > 0) (void)mbar_wait(&sh.cmt_bar, (sh.cmt_issued - 1) & 1, wait_ns);
  if (tid == 0 && sh.st_issued > 0) (void)mbar_wait(&sh.st_bar, (sh.st_issued - 1) & 1, wait_ns);
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

bool pending_commit_tc_supported(const tgdn_tree& prev, const void* prev_k) {
  return prev.depth_max + 1 <= kTcPath && (reinterpret_cast<uintptr_t>(prev_k) % 16) == 0;
}

bool verify_tc_supported(const tgdn_tree& t, const tgdn_dims& d, const void* q, const void* k,
                         const void* v, const float* S0, const void* o, bool small_only) {
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
  return d.io == TGDN_BF16 && d.d_k == kTcDK && d.d_v == kTcDV &&
         (small_only || t.n_max <= kTcNodes) && t.depth_max <= kTcDepth && al(q, 16) &&
         al(k, 16) && al(v, 16) && al(S0, 16) && al(o, 16);
}


cudaError_t launch_verify_tc(const tgdn_tree& t, const tgdn_dims& d, const CUtensorMap& qmap,
                             const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const OutMaps& om, const float* g, const float* b, float* S,
                             void* o, float* U, float* G, const PendingCommit& cm,
                             bool small_only, cudaStream_t s) {
  // the path solve keeps depth_max + 1 partial sums in registers
  auto kern = t.depth_max <= 16 ? verify_tc_kernel<16> : verify_tc_kernel<kTcDepth>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (e != cudaSuccess) return e;
  const long items = (long)t.B * d.H_v;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  const int sms = device_sm_count();
  const int grid = (int)(items < sms ? items : sms);
  // programmatic stream serialization: the kernel's prologue may overlap the
  // previous kernel's tail (it waits for that kernel before reading any input)
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid);
  lc.blockDim = dim3(kTcThreads);
  lc.dynamicSmemBytes = kTcSmemBytes;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  const WaitHooks hk = wait_hooks();
  e = cudaLaunchKernelEx(&lc, kern, qmap, kmap, vmap, om, (int)items, d.H_qk, d.H_v, t.depth_max,
                         t.words, small_only ? 1 : 0, (small_only && t.B <= kMaxCompact) ? 1 : 0,
                         t.cu_nodes, t.depth, t.order, t.pos,
                         t.anc, t.status, g, b, S, static_cast<__nv_bfloat16*>(o), U, G, cm,
                         hk.wait_ns ? hk.wait_ns : kWaitLimitNs, hk.hold_item);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tgdn
