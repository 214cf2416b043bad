// tree_attn.cu — ancestor-masked tree attention on tensor cores (bf16, d = 128).
//
// "Trees from Marginals" (Technisches Resümee, Problemstellung): in attention
// layers a draft tree is verified with an attention mask, each node seeing the
// sequence's cached context and its own root path.  The hybrid verifier's
// attention layers run this on the same trees as its GDN layers, with the same
// ancestor-or-self bitmasks from tree prep.
//
// One CTA per (sequence, key/value head, tile of 128 query rows); a query row
// is (node, query head of the group), row = node * G + g.  256 softmax threads,
// two per row (= TMEM lane), each taking half of every key tile and half of the
// output columns; the halves of a row's maximum are exchanged per tile between
// the two warps that hold the row, and its normaliser merged once at the end.
// Two more warps own no rows: lane 0 of one issues every tensor-core product,
// lane 0 of the other every copy, so the softmax warps never wait for an issuing
// thread among them and the products do not wait behind the copies.  One CTA per SM
// (the 512 TMEM columns: two 128-column score buffers and the 128-column O).
//
// Keys come in tiles of 128: first the cached context (prefix_len[b] positions),
// then the tree's own nodes.  One pass over the key tiles with an online
// softmax: P = exp(logit - m) is formed against a running row maximum m as a
// bf16 operand and O += P V accumulates in TMEM; m is moved (and O, the running
// sum rescaled in place) only when a tile's maximum exceeds it by more than
// kRescaleGap, so P stays below e^kRescaleGap and rescaling is rare.  O is
// divided by the sum at the end.  Pipeline: the score product of tile u + 1
// runs while the softmax warps form P for tile u; P goes to TMEM over its own
// score columns (two score buffers) and is the A operand of O += P V straight
// from TMEM, issued once every softmax warp has arrived on the tile's "P ready"
// barrier.  Key tiles have three buffers and value tiles two, with separate
// barriers: a key buffer is refilled once its score product is done (three tiles
// ahead: with two, the key copy was the chain that set the pace), a value buffer
// once its P V product is done.  The tile is 128 keys wide because
// the SM issues tcgen05.mma instructions at a bounded rate: a 128-key score
// product is 8 instructions of N = 128, where two 64-key tiles took 16 of N = 64.
//
// With a workspace the cached context of each (sequence, head, row tile) is
// split over several CTAs (the tree's own keys go to the last one); each writes
// its unnormalised O, row maximum and sum, and tree_attn_combine_kernel merges
// them (O = sum_s e^{m_s - M} O_s / sum_s e^{m_s - M} l_s).  That keeps every SM
// busy when there are fewer (sequence, head, row tile) items than SMs.
//   S tile = Q K^T: tcgen05.mma, A = Q (TMA, 128-byte swizzle), B = K tile
//   O     += P V:   A = P (bf16 pairs in TMEM), B = V tile (MN-major)
// Every wait is bounded; on expiry the sequence is marked TGDN_SEQ_TIMEOUT.
#include "tgdn_device.cuh"
#include "tgdn_kernels.h"

namespace tgdn {

constexpr int kAtThreads = 256;          // softmax threads: two per query row
constexpr int kAtIssueWarp = kAtThreads / 32;  // the warp that issues every product
constexpr int kAtCopyWarp = kAtIssueWarp + 1;  // the warp that issues every copy
constexpr int kAtBlock = kAtThreads + 64;
constexpr int kAtRows = 128;             // query rows per CTA
constexpr float kRescaleGap = 8.f;       // lazy rescaling threshold (natural log units)
constexpr int kAtKeys = 128;             // keys per tile
constexpr int kAtD = 128;
constexpr int kPartStride = kAtD + 4;    // workspace row: O (128), m, l, 2 pad (528 B, 16-B aligned)
constexpr int kAtMaxNodes = 128;         // tree nodes per sequence on this kernel
constexpr uint32_t kAtTmemCols = 512;    // S / P buffers: cols 0-127, 256-383; O: cols 128-255
constexpr int kAtTileBytes = kAtKeys * 128;  // one d half (or atom) of a key or value tile
constexpr int kAtOffQ = 0;               // [2 d halves][128 rows][128 B]      32 KiB
constexpr int kAtKStages = 3;            // key tiles in flight (value tiles: 2)
constexpr int kAtOffK = 32768;           // 3 x [2 d halves][128 keys][128 B]  3 x 32 KiB
constexpr int kAtOffV = kAtOffK + kAtKStages * 32768;  // 2 x [2 d atoms][128 keys][128 B]
constexpr int kAtOffMask = kAtOffV + 2 * 32768;  // [kAtMaxNodes][2] uint64      2 KiB
constexpr int kAtOffStat = kAtOffMask + kAtMaxNodes * 16;  // [2 tiles][2][128] row max, [2][128] sum
constexpr int kAtOffBar = kAtOffStat + 6 * kAtRows * 4;
// (before the first tile the statistics area holds the copies of the topological order
// and of every position's ancestor masks that the mask build reads)
static_assert(kAtMaxNodes * 4 + kAtMaxNodes * 2 * 8 <= 6 * kAtRows * 4,
              "order and mask copies fit the statistics area");
constexpr int kAtSmemBytes = kAtOffBar + 128 + 1024;
static_assert(kAtSmemBytes <= 227 * 1024, "fits one CTA per SM");

__device__ __forceinline__ int at_swz(int row, int chunk) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4);
}

struct AtArgs {
  int H_q, H_kv, G, n_max, P_max, mtiles, n_items, splits;
  float* part;  // with splits > 1: [splits][n_items][128 rows][kPartStride] = O, m, l, pad
  float scale;
  const int32_t* cu;
  const int32_t* order;
  const int32_t* pos;
  const uint64_t* anc;
  int words;
  int32_t* status;
  const int32_t* prefix_len;
  __nv_bfloat16* o;
};

__global__ void __launch_bounds__(kAtBlock, 1)
tree_attn_kernel(const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap ktmap,
                 const __grid_constant__ CUtensorMap vtmap,
                 const __grid_constant__ CUtensorMap kcmap,
                 const __grid_constant__ CUtensorMap vcmap, const AtArgs a) {
  extern __shared__ uint8_t at_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* amask = reinterpret_cast<uint64_t*>(smem + kAtOffMask);
  uint64_t* kbar = reinterpret_cast<uint64_t*>(smem + kAtOffBar);  // [3] key tile (+ Q)
  uint64_t* vbar = kbar + kAtKStages;  // [2] value tile
  uint64_t* sbar = vbar + 2;     // [2] score product of tile u (buffer u & 1)
  uint64_t* pvbar = sbar + 2;    // [2] P V product of tile u
  uint64_t* pready = pvbar + 2;  // [2] P of tile u in TMEM: one arrival per softmax warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pready + 2);
  int* s_abort = reinterpret_cast<int*>(tmem_slot + 1);

  const int item = blockIdx.x / a.splits, sp = blockIdx.x % a.splits;
  if (item >= a.n_items) return;
  const int mt = item % a.mtiles;
  const int hk = (item / a.mtiles) % a.H_kv;
  const int b = item / (a.mtiles * a.H_kv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the sequence's bounds, status and context length in one round trip
  const int c0 = a.cu[b], c1 = a.cu[b + 1], st_b = a.status[b], pl_b = a.prefix_len[b];
  const int lo = c0, N = c1 - c0;
  const int npt = kAtRows / a.G;             // nodes per tile of query rows
  const int node0 = mt * npt;
  if (N <= 0 || node0 >= N) return;          // no rows of this tile exist
  if (st_b == TGDN_SEQ_BAD_RANGE) return;  // rows outside the arrays: untouched
  const int row = tid & (kAtRows - 1), kh = tid >> 7;  // TMEM lane; key / column half
  const int my_node = node0 + row / a.G, my_g = row % a.G;
  const bool row_live = my_node < N;
  __nv_bfloat16* orow =
      a.o + ((size_t)(lo + my_node) * a.H_q + hk * a.G + my_g) * kAtD;
  if (st_b != TGDN_SEQ_OK || N > kAtMaxNodes || N > a.n_max) {
    if (row_live && tid < kAtThreads)
      for (int c = kh * 8; c < kh * 8 + 8; ++c)
        reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
    return;
  }
  const int P = max(0, min(pl_b, a.P_max));

  if (tid == 0) {
    for (int i = 0; i < kAtKStages; ++i) mbar_init(&kbar[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&vbar[i], 1);
      mbar_init(&sbar[i], 1);
      mbar_init(&pvbar[i], 1);
      mbar_init(&pready[i], kAtThreads / 32);
    }
    fence_mbar_init();
    *s_abort = 0;
  }
  const int nt_pre = (P + kAtKeys - 1) / kAtKeys;
  const int nt_tree = (N + kAtKeys - 1) / kAtKeys;
  // this CTA's key tiles: context tiles [t_begin, t_end), then (last split) the tree's
  const int t_begin = (int)(((long)sp * nt_pre) / a.splits);
  const int t_end = (int)(((long)(sp + 1) * nt_pre) / a.splits);
  const int n_ctx = t_end - t_begin;
  const int nt = n_ctx + (sp == a.splits - 1 ? nt_tree : 0);  // steps of this CTA
  auto tile_of = [&](int u) { return u < n_ctx ? t_begin + u : nt_pre + (u - n_ctx); };

  // Steps u = 0 .. nt - 1: key tile u in buffer u % 3, value tile u in buffer u & 1,
  // scores and P in TMEM buffer u & 1.  Lane 0 of the copy warp issues every copy and
  // lane 0 of the product warp every product; no waiter can be a whole phase behind.
  int k_issued[kAtKStages] = {0, 0, 0}, v_issued[2] = {0, 0};  // copies issued per buffer
  int s_issued[2] = {0, 0}, pv_issued[2] = {0, 0};  // products issued per barrier
  auto tile_row = [&](int u, const CUtensorMap*& km, const CUtensorMap*& vm) {
    const int t = tile_of(u);
    const bool pre = t < nt_pre;
    km = pre ? &kcmap : &ktmap;
    vm = pre ? &vcmap : &vtmap;
    return pre ? b * a.P_max + t * kAtKeys : lo + (t - nt_pre) * kAtKeys;
  };
  auto issue_k = [&](int u) {  // key tile u (with Q for u = 0) into key buffer u % 3
    const CUtensorMap *km, *vm;
    const int r = tile_row(u, km, vm);
    uint64_t* bar = &kbar[u % kAtKStages];
    mbar_arrive_expect_tx(bar, 2 * kAtKeys * 128 + (u == 0 ? 32768 : 0));
    if (u == 0) {
      tma_load_3d(smem + kAtOffQ, &qmap, bar, 0, hk * a.G, lo + node0);
      tma_load_3d(smem + kAtOffQ + 16384, &qmap, bar, 64, hk * a.G, lo + node0);
    }
    uint8_t* kdst = smem + kAtOffK + (u % kAtKStages) * (2 * kAtTileBytes);
    tma_load_3d(kdst, km, bar, 0, hk, r);
    tma_load_3d(kdst + kAtTileBytes, km, bar, 64, hk, r);
    k_issued[u % kAtKStages] += 1;
  };
  auto issue_v = [&](int u) {  // value tile u into value buffer u & 1
    const CUtensorMap *km, *vm;
    const int r = tile_row(u, km, vm);
    uint64_t* bar = &vbar[u & 1];
    mbar_arrive_expect_tx(bar, 2 * kAtKeys * 128);
    uint8_t* vdst = smem + kAtOffV + (u & 1) * (2 * kAtTileBytes);
    tma_load_3d(vdst, vm, bar, 0, hk, r);
    tma_load_3d(vdst + kAtTileBytes, vm, bar, 64, hk, r);
    v_issued[u & 1] += 1;
  };

  // ancestor-or-self sets in node-index space (bit s of word s / 64).  The topological
  // order goes to shared memory first (one coalesced load), so that the bit loop does
  // not wait a global-memory round trip per ancestor.
  // The topological order and the ancestor masks of every position go to shared memory
  // first (one round trip, issued before the first tiles' copies), so that no load waits
  // behind those copies and the bit loop waits no round trip per ancestor.
  int* sord = reinterpret_cast<int*>(smem + kAtOffStat);  // free until the first tile
  uint64_t* sanc = reinterpret_cast<uint64_t*>(smem + kAtOffStat + kAtMaxNodes * 4);  // [pos][2]
  int p_anc = -1, ord_v = -1;
  uint64_t anc_v[2] = {0ull, 0ull};
  if (tid < N) {
    ord_v = a.order[lo + tid];
    p_anc = a.pos[lo + tid];
    for (int w = 0; w < a.words && w < 2; ++w) anc_v[w] = a.anc[(size_t)(lo + tid) * a.words + w];
  }
  if (warp == 0) tmem_alloc(tmem_slot, kAtTmemCols);
  __syncthreads();
  // the first key and value tiles (and Q) go out while the masks are built
  if (warp == kAtCopyWarp && lane == 0 && nt > 0) {
    issue_k(0);
    issue_v(0);
    if (nt > 1) {
      issue_k(1);
      issue_v(1);
    }
    if (nt > 2) issue_k(2);
  }
  if (tid < N) {
    sord[tid] = ord_v;
    sanc[2 * tid] = anc_v[0];
    sanc[2 * tid + 1] = anc_v[1];
  }
  __syncthreads();
  if (tid < N) {
    uint64_t m0 = 0, m1 = 0;
    const int p = p_anc;
    if (p >= 0 && p < N) {
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        uint64_t bits = sanc[2 * p + w];
        while (bits) {
          const int bp = w * 64 + __ffsll(static_cast<long long>(bits)) - 1;
          bits &= bits - 1;
          const int s = bp < N ? sord[bp] : -1;
          if (s >= 0 && s < 64) m0 |= 1ull << s;
          else if (s >= 64 && s < 128) m1 |= 1ull << (s - 64);
        }
      }
    }
    amask[2 * tid] = m0;
    amask[2 * tid + 1] = m1;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 128;
  auto tS_of = [&](int u) -> uint32_t { return tmem + ((u & 1) ? 256u : 0u); };
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  volatile int* abort = s_abort;

  const uint64_t m_lo = row_live ? amask[2 * my_node] : 0;
  const uint64_t m_hi = row_live ? amask[2 * my_node + 1] : 0;
  // S = Q K^T of tile u into score buffer u & 1 (once its key tile has landed)
  auto score = [&](int u) -> bool {
    if (!mbar_wait_suspend(&kbar[u % kAtKStages], (u / kAtKStages) & 1, abort)) return false;
    tc_fence_after_sync();
    const uint32_t sQ = smem_addr(smem + kAtOffQ);
    const uint32_t sK = smem_addr(smem + kAtOffK + (u % kAtKStages) * (2 * kAtTileBytes));
    constexpr uint32_t id_s = idesc_bf16_f32(128, kAtKeys, 0, 0);
#pragma unroll
    for (int s = 0; s < kAtD / 16; ++s) {
      const uint64_t ad = smem_desc(sQ + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024, kSwizzle128B);
      const uint64_t bd =
          smem_desc(sK + (s >> 2) * kAtTileBytes + (s & 3) * 32, 16, 1024, kSwizzle128B);
      umma_bf16(tS_of(u), ad, bd, id_s, s > 0);
    }
    umma_commit(&sbar[u & 1]);
    s_issued[u & 1] += 1;
    return true;
  };
  // this thread's 64 raw scores q.k of tile u (keys kh * 64 ..), masked to -inf
  // (the softmax scale enters with the exponent; only a partial context tile, a
  // row past the tree or a tree tile needs the mask)
  constexpr int kHalf = kAtKeys / 2;
  auto read_logits = [&](int u, float (&x)[kHalf]) {
    const int t = tile_of(u);
#pragma unroll
    for (int q = 0; q < kHalf / 32; ++q) {
      float y[32];
      tmem_ld32(tS_of(u) + lane_base + kh * kHalf + q * 32, y);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; ++c) x[q * 32 + c] = y[c];
    }
    if (t < nt_pre) {
      const int lim = P - t * kAtKeys - kh * kHalf;  // keys below lim are cached context
      if (lim < kHalf || !row_live) {
#pragma unroll
        for (int c = 0; c < kHalf; ++c)
          if (c >= lim || !row_live) x[c] = -INFINITY;
      }
    } else {
      const int s0 = (t - nt_pre) * kAtKeys + kh * kHalf;
      const uint64_t mk = (s0 < 64 ? m_lo : m_hi) >> (s0 & 63);
#pragma unroll
      for (int c = 0; c < kHalf; ++c)
        if (s0 + c >= N || !((mk >> c) & 1ull)) x[c] = -INFINITY;
    }
  };

  bool ok = true;
  float* st = reinterpret_cast<float*>(smem + kAtOffStat);
  float m = -INFINITY;  // running maximum of the row's raw scores (same in both threads)
  // exp(scale (x - m)) = 2^(x c - m c) with c = scale log2(e); the rescaling
  // threshold kRescaleGap (natural-log units) in raw-score units
  const float c2 = a.scale * 1.4426950408889634f;
  const float gap_raw = kRescaleGap / a.scale;
  float lsum = 0.f;     // this thread's half of the row's sum of exp(logit - m)
  if (warp == kAtCopyWarp) {
    // ---- the copy warp: key tile u + 3 into key buffer u % 3 once S(u) is done,
    // value tile u + 2 into value buffer u & 1 once P V of tile u is done (a key tile
    // is requested three tiles ahead: its copy, not the products, was the chain that
    // set the pace with two key buffers)
    if (lane == 0 && nt > 0) {
      for (int u = 0; ok && u + 2 < nt; ++u) {
        const uint32_t ph = (u >> 1) & 1;
        ok = mbar_wait_suspend(&sbar[u & 1], ph, abort);
        if (ok && u + 3 < nt) issue_k(u + 3);
        if (ok) ok = mbar_wait_suspend(&pvbar[u & 1], ph, abort);
        if (ok) issue_v(u + 2);
      }
    }
    __syncwarp();
  } else if (warp == kAtIssueWarp) {
    // ---- the product warp: S(u + 1) is issued while the softmax warps form P of
    // tile u, then O += P V of tile u once every softmax warp has stored its P
    if (lane == 0 && nt > 0) {
      ok = score(0);
      for (int u = 0; ok && u < nt; ++u) {
        const uint32_t ph = (u >> 1) & 1;
        if (u + 1 < nt) {
          // P V of tile u - 1 is done: score buffer (u + 1) & 1 is free
          if (u > 0) ok = mbar_wait_suspend(&pvbar[(u - 1) & 1], ((u - 1) >> 1) & 1, abort);
          if (ok) ok = score(u + 1);
        }
        if (ok) ok = mbar_wait_suspend(&pready[u & 1], ph, abort);
        if (ok) ok = mbar_wait_suspend(&vbar[u & 1], ph, abort);
        if (ok) {  // O += P V: A = P from TMEM (16 keys = 8 columns per step)
          tc_fence_after_sync();
          const uint32_t sV = smem_addr(smem + kAtOffV + (u & 1) * (2 * kAtTileBytes));
          constexpr uint32_t id_o = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll
          for (int s = 0; s < kAtKeys / 16; ++s) {
            // MN-major V: the two 64-column atoms one tile half apart, 8-key groups 1 KiB apart
            const uint64_t bd = smem_desc(sV + s * 2048, kAtTileBytes, 1024, kSwizzle128B);
            umma_bf16_tmem_a(tO, tS_of(u) + s * 8, bd, id_o, (u > 0 || s > 0) ? 1u : 0u);
          }
          umma_commit(&pvbar[u & 1]);
          pv_issued[u & 1] += 1;
        }
      }
      // the last P V product: O is final
      if (ok) ok = mbar_wait_suspend(&pvbar[(nt - 1) & 1], ((nt - 1) >> 1) & 1, abort);
    }
    __syncwarp();
  } else {
    // ---- softmax warps.  The two threads of a row sit in warps w and w + 4 (the
    // same TMEM lane quarter); they exchange their halves' maxima through shared
    // memory behind a barrier of that warp pair, which also carries the decision
    // to stop (so both warps of a pair leave the loop at the same step).
    const int pair_bar = 1 + (warp & 3);
    for (int u = 0; u < nt; ++u) {
      const uint32_t ph = (u >> 1) & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait_suspend(&sbar[u & 1], ph, abort)) != 0;
      float x[kHalf];
      float lm = -INFINITY;
      if (ok) {
        tc_fence_after_sync();
        read_logits(u, x);
        // pairwise: five dependent levels instead of 31
        float t[kHalf / 2];
#pragma unroll
        for (int c = 0; c < kHalf / 2; ++c) t[c] = fmaxf(x[2 * c], x[2 * c + 1]);
#pragma unroll
        for (int w = kHalf / 4; w >= 1; w /= 2)
#pragma unroll
          for (int c = 0; c < w; ++c) t[c] = fmaxf(t[c], t[c + w]);
        lm = t[0];
      }
      float* stu = st + (u & 1) * 2 * kAtRows;
      stu[kh * kAtRows + row] = lm;
      // (also: both halves of the row have read their scores before P overwrites them)
      if (!named_sync_and(pair_bar, 64, ok && !*abort)) {
        ok = false;
        break;
      }
      const float mt = fmaxf(stu[row], stu[kAtRows + row]);
      const bool need = mt > m + gap_raw;  // also the first finite maximum of the row
      const float alpha = need ? (m == -INFINITY ? 0.f : fast_exp2((m - mt) * c2)) : 1.f;
      if (need) {
        m = mt;
        lsum *= alpha;
      }
      if (u > 0 && __any_sync(0xffffffffu, need)) {  // O *= alpha (warp-collective)
        // O is stable once the previous tile's P V product is done
        ok = __all_sync(0xffffffffu,
                        mbar_wait_suspend(&pvbar[(u - 1) & 1], ((u - 1) >> 1) & 1, abort)) != 0;
        if (ok) {
          tc_fence_after_sync();
#pragma unroll 1
          for (int q = 4 * kh; q < 4 * kh + 4; ++q) {  // 16 columns at a time
            float r[16];
            tmem_ld16(tO + lane_base + q * 16, r);
            tmem_ld_wait();
            uint32_t w[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) w[c] = __float_as_uint(r[c] * alpha);
            tmem_st16(tO + lane_base + q * 16, w);
          }
        }
      }
      if (!ok) continue;  // the next pair barrier stops both warps
      // P = exp(logit - m) as bf16 pairs over this thread's 32 score columns' first
      // 16 (key 2 c and 2 c + 1 in column c of the half)
      // (m = -inf only while every score so far is masked: then 2^(-inf) = 0)
      const float mc = m == -INFINITY ? 0.f : m * c2;
      uint32_t pw[kHalf / 2];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};  // four independent partial sums
#pragma unroll
      for (int i = 0; i < kHalf / 2; ++i) {
        const float p0 = fast_exp2(fmaf(x[2 * i], c2, -mc));
        const float p1 = fast_exp2(fmaf(x[2 * i + 1], c2, -mc));
        ps[i & 3] += p0 + p1;
        const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
        pw[i] = *reinterpret_cast<const uint32_t*>(&pp);
      }
      lsum += (ps[0] + ps[1]) + (ps[2] + ps[3]);
#pragma unroll
      for (int q = 0; q < kHalf / 32; ++q) {
        uint32_t w16[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) w16[c] = pw[q * 16 + c];
        tmem_st16(tS_of(u) + lane_base + kh * (kHalf / 2) + q * 16, w16);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[u & 1]);
    }
  }
  ok = __syncthreads_and(ok) != 0;
  // the row's sum from its two halves (both kept against the same maximum)
  float* ssum = st + 4 * kAtRows;
  if (tid < kAtThreads) ssum[kh * kAtRows + row] = lsum;
  __syncthreads();
  const float l = tid < kAtThreads ? ssum[row] + ssum[kAtRows + row] : 0.f;
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  // ---- epilogue: O rows to global (bf16), or this split's part to the workspace
  if (tid >= kAtThreads) {
    if (!ok && lane == 0) {
      // an expired wait: report it, and let the latest copies and products land (bounded)
      atomicCAS(&a.status[b], TGDN_SEQ_OK, TGDN_SEQ_TIMEOUT);
      for (int bf = 0; bf < kAtKStages; ++bf)
        if (k_issued[bf] > 0) (void)mbar_wait(&kbar[bf], (k_issued[bf] - 1) & 1);
      for (int bf = 0; bf < 2; ++bf) {
        if (v_issued[bf] > 0) (void)mbar_wait(&vbar[bf], (v_issued[bf] - 1) & 1);
        if (s_issued[bf] > 0) (void)mbar_wait(&sbar[bf], (s_issued[bf] - 1) & 1);
        if (pv_issued[bf] > 0) (void)mbar_wait(&pvbar[bf], (pv_issued[bf] - 1) & 1);
      }
    }
  } else if (ok && a.splits > 1) {
    tc_fence_after_sync();
    float* prow = a.part + (((size_t)sp * a.n_items + item) * kAtRows + row) * kPartStride;
#pragma unroll
    for (int q = 2 * kh; q < 2 * kh + 2; ++q) {
      float r[32];
      tmem_ld32(tO + lane_base + q * 32, r);
      tmem_ld_wait();
      if (nt == 0) {
#pragma unroll
        for (int c = 0; c < 32; ++c) r[c] = 0.f;
      }
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4)
        *reinterpret_cast<float4*>(prow + q * 32 + c4 * 4) =
            make_float4(r[c4 * 4], r[c4 * 4 + 1], r[c4 * 4 + 2], r[c4 * 4 + 3]);
    }
    if (kh == 0) {
      prow[kAtD] = m * a.scale;  // the row maximum of the scaled logits
      prow[kAtD + 1] = l;
    }
  } else if (ok) {
    tc_fence_after_sync();
#pragma unroll
    for (int q = 2 * kh; q < 2 * kh + 2; ++q) {  // this thread's 64 output columns
      float r[32];
      tmem_ld32(tO + lane_base + q * 32, r);
      tmem_ld_wait();
      if (row_live) {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 pp = __floats2bfloat162_rn(r[c8 * 8 + 2 * i] * inv_l,
                                                            r[c8 * 8 + 2 * i + 1] * inv_l);
            w[i] = *reinterpret_cast<const uint32_t*>(&pp);
          }
          reinterpret_cast<uint4*>(orow)[q * 4 + c8] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kAtTmemCols);
  }
}

// Merges the context splits of one (sequence, key/value head, row tile) item:
// 256 threads, two per row (64 output columns each).
__global__ void __launch_bounds__(kAtThreads)
tree_attn_combine_kernel(const AtArgs a) {
  const int item = blockIdx.x;
  const int mt = item % a.mtiles;
  const int hk = (item / a.mtiles) % a.H_kv;
  const int b = item / (a.mtiles * a.H_kv);
  const int tid = threadIdx.x;
  const int lo = a.cu[b], N = a.cu[b + 1] - lo;
  const int node0 = mt * (kAtRows / a.G);
  if (N <= 0 || node0 >= N || a.status[b] != TGDN_SEQ_OK) return;  // zeros already written
  const int row = tid & (kAtRows - 1), kh = tid >> 7;
  const int my_node = node0 + row / a.G, my_g = row % a.G;
  if (my_node >= N) return;
  const size_t stride = (size_t)a.n_items * kAtRows * kPartStride;
  const float* p0 = a.part + ((size_t)item * kAtRows + row) * kPartStride;
  float M = -INFINITY;
  for (int s = 0; s < a.splits; ++s) M = fmaxf(M, p0[s * stride + kAtD]);
  float L = 0.f, acc[64];
#pragma unroll
  for (int c = 0; c < 64; ++c) acc[c] = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const float* ps = p0 + s * stride;
    const float ms = ps[kAtD];
    if (ms == -INFINITY) continue;  // no visible key in this split
    const float w = __expf(ms - M);
    L = fmaf(w, ps[kAtD + 1], L);
#pragma unroll
    for (int c4 = 0; c4 < 16; ++c4) {
      const float4 x = reinterpret_cast<const float4*>(ps + kh * 64)[c4];
      acc[c4 * 4] = fmaf(w, x.x, acc[c4 * 4]);
      acc[c4 * 4 + 1] = fmaf(w, x.y, acc[c4 * 4 + 1]);
      acc[c4 * 4 + 2] = fmaf(w, x.z, acc[c4 * 4 + 2]);
      acc[c4 * 4 + 3] = fmaf(w, x.w, acc[c4 * 4 + 3]);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint4* orow = reinterpret_cast<uint4*>(
      a.o + ((size_t)(lo + my_node) * a.H_q + hk * a.G + my_g) * kAtD + kh * 64);
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 pp =
          __floats2bfloat162_rn(acc[c8 * 8 + 2 * i] * inv, acc[c8 * 8 + 2 * i + 1] * inv);
      w[i] = *reinterpret_cast<const uint32_t*>(&pp);
    }
    orow[c8] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}


// Context splits for this launch: enough CTAs for one per SM, at most 8, and at
// least 1024 cached positions per split, below which the merge costs more than the
// split saves.
static int attn_splits(const tgdn_tree& t, int H_q, int H_kv, int P_max) {
  const int G = H_q / H_kv;
  const long items = (long)t.B * H_kv * ((t.n_max * G + kAtRows - 1) / kAtRows);
  if (items <= 0) return 1;
  long s = (long)device_sm_count() / items;
  const long ctx_tiles = (P_max + kAtKeys - 1) / kAtKeys;
  if (s > 8) s = 8;
  if (s > ctx_tiles / (1024 / kAtKeys)) s = ctx_tiles / (1024 / kAtKeys);
  return s < 1 ? 1 : (int)s;
}

size_t tree_attn_workspace_bytes(const tgdn_tree& t, int H_q, int H_kv, int P_max) {
  const int splits = attn_splits(t, H_q, H_kv, P_max);
  if (splits <= 1) return 0;
  const int G = H_q / H_kv;
  const size_t items = (size_t)t.B * H_kv * ((t.n_max * G + kAtRows - 1) / kAtRows);
  return (size_t)splits * items * kAtRows * kPartStride * sizeof(float);
}

bool tree_attn_supported(const tgdn_tree& t, int H_q, int H_kv, int d) {
  const int G = H_kv > 0 ? H_q / H_kv : 0;
  return d == kAtD && H_kv > 0 && H_q % H_kv == 0 && (G == 1 || G == 2 || G == 4 || G == 8 ||
                                                      G == 16) &&
         t.n_max <= kAtMaxNodes;
}

cudaError_t launch_tree_attn(const tgdn_tree& t, int H_q, int H_kv, int P_max, float scale,
                             const CUtensorMap& qmap, const CUtensorMap& ktmap,
                             const CUtensorMap& vtmap, const CUtensorMap& kcmap,
                             const CUtensorMap& vcmap, const int32_t* prefix_len, void* o,
                             void* ws, size_t ws_bytes, cudaStream_t s) {
  AtArgs a;
  a.H_q = H_q;
  a.H_kv = H_kv;
  a.G = H_q / H_kv;
  a.n_max = t.n_max;
  a.P_max = P_max;
  a.mtiles = (t.n_max * a.G + kAtRows - 1) / kAtRows;
  const long items = (long)t.B * H_kv * a.mtiles;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  a.n_items = (int)items;
  a.scale = scale;
  a.cu = t.cu_nodes;
  a.order = t.order;
  a.pos = t.pos;
  a.anc = t.anc;
  a.words = t.words;
  a.status = t.status;
  a.prefix_len = prefix_len;
  a.o = static_cast<__nv_bfloat16*>(o);
  const size_t need = tree_attn_workspace_bytes(t, H_q, H_kv, P_max);
  a.splits = (need > 0 && ws != nullptr && ws_bytes >= need) ? attn_splits(t, H_q, H_kv, P_max)
                                                              : 1;
  a.part = a.splits > 1 ? static_cast<float*>(ws) : nullptr;
  if ((long)a.n_items * a.splits > 0x7fffffffL) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(tree_attn_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kAtSmemBytes);
  if (e != cudaSuccess) return e;
  // the whole unified L1 / shared memory as shared memory
  e = cudaFuncSetAttribute(tree_attn_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  tree_attn_kernel<<<(unsigned)(items * a.splits), kAtBlock, kAtSmemBytes, s>>>(
      qmap, ktmap, vtmap, kcmap, vcmap, a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  tree_attn_combine_kernel<<<(unsigned)items, kAtThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tgdn
