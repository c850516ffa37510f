// Device-side batch plan: turns (query_start_loc, seq_lens) into the list of
// work items the scoring kernel walks, without any host round trip.
//
// A work item is (request r, a group of up to G consecutive query rows of r,
// a key range [k0, k1) of r's context).  Groups of rows share every key tile
// they load (the rows' heads are the N side of one MMA).
//
// Balance: the groups' key tiles (128 keys each) are laid end to end, W tiles
// in all, and CTA c of the n_cta persistent CTAs takes the tiles
// [c*Q, (c+1)*Q) with Q = max(ceil(W / n_cta), min_tiles).  A group that
// straddles a CTA boundary is cut there into pieces ("splits") that run on
// different CTAs; each piece keeps a superset of its rows' top-k and the last
// piece of a group to finish merges them.  CTA c walks the items
// [cta_start[c], cta_start[c+1]).
#pragma once

#include <cstdint>

#include "kwrite.cuh"

namespace dsa {

struct Item {
  int32_t r;           // request
  int32_t t0;          // first query row of the group
  int32_t gcount;      // rows in the group (1..G)
  int32_t k0, k1;      // key range [k0, k1) (logical positions); k0 % 128 == 0
  int32_t split;       // piece index | (number of pieces << 16)
  int32_t cand_block;  // first candidate block of the group (split groups), else -1
  int32_t sgroup;      // split-group id (index of its done counter), -1, or kSgroupRows
};
constexpr int32_t kSgroupRows = -2;  // the item's row is scored into the workspace
static_assert(sizeof(Item) == 32, "Item must stay 32 bytes");

// Per scoring CTA: its item range and a copy of its first item, so that the
// kernel reaches its first item's pages in two dependent loads, not three.
struct CtaHead {
  Item first;        // valid when it_begin < it_end
  int32_t it_begin;  // = cta_start[c]
  int32_t it_end;    // = cta_start[c + 1]
  int32_t pad[2];
};
static_assert(sizeof(CtaHead) == 48, "CtaHead must stay 48 bytes");

constexpr int kMaxCtas = 320;       // upper bound on the scoring grid (one CTA per SM)
constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemRequests = 4096;  // group prefix held in shared memory up to this many requests
constexpr int kTileKeysPlan = 128;  // keys per tile, the unit of the balance

struct PlanHeader {
  int32_t n_items;
  int32_t n_split_groups;
  int32_t n_cand_blocks;
  int32_t tiles_per_cta;
  int32_t total_groups;
  int32_t n_used_ctas;
  int32_t pad[58];
};
static_assert(sizeof(PlanHeader) == 256, "PlanHeader is one 256-byte line");

// Candidate-block capacity of one row of one piece: the piece's top-k plus
// room for the rest of the level-1 bin that holds its k-th largest key.
__host__ __device__ inline int cand_block_capacity(int k) {
  const int c = k + (k < 1024 ? k : 1024);
  return (c + 31) / 32 * 32;
}

// Workspace carve-up; identical on host and device.
constexpr int kBlockBins = 2048;  // level-1 bins published with every candidate block

// Decode batches (one query row per group) may score their rows into the
// workspace instead and select each row's top-k with a second kernel: the
// scoring kernel then streams keys without selecting, splitting or merging.
// A row takes that path when it sees at most score_stride keys (a multiple of
// 128, at most kScoreRowMax; 0 = never).
constexpr int kScoreRowMax = 8192;   // longer rows merge faster across SMs (measured)

// A decode row (one row per group) cut into at least this many pieces is
// "wide": its pieces share two level-1 histograms of its keys (see the
// scoring kernel's epilogue): one they publish early to bound the row's k-th
// score, and one of their final candidates for the merge.  A wide group spends
// kWideSplit - 1 of the n_cta - 1 CTA boundaries, which bounds their number.
// (A finer early histogram -- 8192 bins of the key's top 13 bits, published
// per candidate -- measured slower: the bound it gives after the first few
// thousand keys of each piece is weaker than the level-1 bound a piece gives
// from a fuller buffer.)
constexpr int kWideSplit = 4;
constexpr int kSharedHistWords = 2 * kBlockBins;  // per wide split group

struct WsLayout {
  size_t header, group_prefix, cta_start, heads, items, done, wide_of, cand_count, cand_keys,
      cand_idx, cand_hist, cand_start, ghist, row_keys, score_rows, total;
  int max_items, max_split_groups, max_cand_blocks, cb, score_stride, max_wide;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// A piece boundary is a CTA boundary inside a group, so at most n_cta - 1 of
// them: at most T + n_cta items, min(n_cta, groups) split groups and
// (split groups + n_cta - 1) pieces of split groups, G candidate blocks each.
// A request of q rows has ceil(q / G) groups, so groups <= min(T, T / G + R).
__host__ __device__ inline WsLayout ws_layout(int T, int R, int G, int k, int n_cta,
                                               int score_stride = 0) {
  WsLayout L;
  L.score_stride = score_stride;
  L.max_items = T + n_cta;
  const long long groups = T < (T + G - 1) / G + R ? T : (T + G - 1) / G + R;
  L.max_split_groups = (int)(groups < n_cta ? groups : n_cta);
  L.max_cand_blocks = G * (L.max_split_groups + n_cta);
  L.cb = cand_block_capacity(k);
  L.max_wide = G == 1 ? (L.max_split_groups < (n_cta - 1) / (kWideSplit - 1)
                             ? L.max_split_groups
                             : (n_cta - 1) / (kWideSplit - 1))
                      : 0;
  size_t o = 0;
  L.header = o;       o = align256(o + sizeof(PlanHeader));
  L.group_prefix = o; o = align256(o + sizeof(int32_t) * (size_t)(R + 1));
  L.cta_start = o;    o = align256(o + sizeof(int32_t) * (size_t)(n_cta + 1));
  L.heads = o;        o = align256(o + sizeof(CtaHead) * (size_t)n_cta);
  L.items = o;        o = align256(o + sizeof(Item) * (size_t)L.max_items);
  L.done = o;         o = align256(o + sizeof(int32_t) * (size_t)L.max_split_groups);
  L.wide_of = o;      o = align256(o + sizeof(int32_t) * (size_t)L.max_split_groups);
  L.cand_count = o;   o = align256(o + sizeof(int32_t) * (size_t)L.max_cand_blocks);
  L.cand_keys = o;    o = align256(o + sizeof(uint32_t) * (size_t)L.max_cand_blocks * L.cb);
  L.cand_idx = o;     o = align256(o + sizeof(int32_t) * (size_t)L.max_cand_blocks * L.cb);
  L.cand_hist = o;    o = align256(o + sizeof(uint16_t) * (size_t)L.max_cand_blocks * kBlockBins);
  L.cand_start = o;   o = align256(o + sizeof(uint16_t) * (size_t)L.max_cand_blocks * kBlockBins);
  L.ghist = o;        o = align256(o + sizeof(uint32_t) * (size_t)L.max_wide * kSharedHistWords);
  L.row_keys = o;     o = align256(o + (score_stride > 0 ? sizeof(int32_t) * (size_t)T : 0));
  L.score_rows = o;   o = align256(o + sizeof(uint32_t) * (size_t)T * (size_t)score_stride);
  L.total = o;
  return L;
}

// Block-wide exclusive scan of one int64 per thread (blockDim.x == kPlanThreads).
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* total,
                                                          long long* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long s = (lane < (kPlanThreads >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const long long warp_off = (warp > 0) ? warp_sums[warp - 1] : 0;
  *total = warp_sums[(kPlanThreads >> 5) - 1];
  __syncthreads();
  return warp_off + x - v;
}

struct PlanParams {
  const int32_t* qsl;
  const int32_t* seq_lens;
  int R, T, G, max_blocks, index_topk;
  int ratio;       // tokens per cache entry (1: plain cache)
  int n_cta;       // CTAs of the scoring launch (<= kMaxCtas)
  int min_tiles;   // smallest per-CTA share worth a piece of its own
  // tiles charged for starting a group's first piece: a CTA's item switch
  // costs its producer about this much streaming time, so the balance counts
  // it and a CTA that holds several items gets fewer keys (< min_tiles)
  int item_cost;
  int32_t* topk_buffer;  // for -1 rows of malformed requests
  unsigned char* ws;
  WsLayout L;
  int32_t* status;
};

// Cache entries visible to the last row of group g of a request with prefix P
// and q new rows: the row at position pos sees (pos + 1) / ratio entries.
__device__ __forceinline__ long long group_keys(long long P, int q, int G, int g, int ratio) {
  const int last = min((g + 1) * G, q);
  return (P + last) / ratio;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
  pdl_launch_dependents();  // the scoring kernel's prologue may overlap the plan
  int32_t* row_keys = reinterpret_cast<int32_t*>(p.ws + p.L.row_keys);
  if (p.L.score_stride > 0)
    for (int t = threadIdx.x; t < p.T; t += kPlanThreads) row_keys[t] = 0;
  __shared__ long long warp_sums[32];
  __shared__ long long s_Q;
  __shared__ unsigned long long s_max_keys;
  __shared__ int2 s_empty[kPlanThreads];  // (first row, rows) of groups that see no entry
  __shared__ int32_t s_wide[kMaxCtas];  // per split group: its wide index, or -1
  __shared__ int s_n_empty;
  // the group prefix of a batch of at most kPlanSmemRequests requests, for the
  // per-group binary search (a search over global memory is a chain of
  // dependent loads, about half a microsecond each)
  __shared__ int32_t s_gp[kPlanSmemRequests + 1];
  const bool gp_in_smem = p.R <= kPlanSmemRequests;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.L.header);
  int32_t* group_prefix = reinterpret_cast<int32_t*>(p.ws + p.L.group_prefix);
  int32_t* cta_start = reinterpret_cast<int32_t*>(p.ws + p.L.cta_start);
  Item* items = reinterpret_cast<Item*>(p.ws + p.L.items);
  int32_t* done = reinterpret_cast<int32_t*>(p.ws + p.L.done);
  const int G = p.G;

  // Phase A: groups per request (prefix sums).
  long long groups_carry = 0;
  for (int base = 0; base < p.R; base += kPlanThreads) {
    const int r = base + threadIdx.x;
    long long groups = 0;
    if (r < p.R) {
      const int qb = p.qsl[r], qe = p.qsl[r + 1];
      const int q = qe - qb, seq = p.seq_lens[r];
      const bool bad = q < 0 || seq < q ||
                       (long long)(seq / p.ratio) > (long long)p.max_blocks * kPageTokens ||
                       qb < 0 || qe > p.T;
      if (bad) {
        raise_status(p.status, kStatusBadMetadata);
        // rows of a malformed request hold no indices
        for (int t = max(qb, 0); t < min(qe, p.T); ++t)
          for (int i = 0; i < p.index_topk; ++i) p.topk_buffer[(size_t)t * p.index_topk + i] = -1;
      } else if (q > 0) {
        groups = (q + G - 1) / G;
      }
    }
    long long tot;
    const long long ex = block_exclusive_scan(groups, &tot, warp_sums);
    if (r < p.R) {
      group_prefix[r] = (int32_t)(groups_carry + ex);
      if (gp_in_smem) s_gp[r] = (int32_t)(groups_carry + ex);
    }
    groups_carry += tot;
  }
  if (threadIdx.x == 0) {
    group_prefix[p.R] = (int32_t)groups_carry;
    if (gp_in_smem) s_gp[p.R] = (int32_t)groups_carry;
  }
  __syncthreads();
  const int32_t* gp = gp_in_smem ? s_gp : group_prefix;
  const int total_groups = (int)groups_carry;

  auto describe = [&](int gi, int& r, int& t0, int& gcount, long long& keys) {
    int lo = 0, hi = p.R - 1;  // last r with group_prefix[r] <= gi
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (gp[mid] <= gi) lo = mid; else hi = mid - 1;
    }
    r = lo;
    const int g = gi - gp[r];
    const int qb = p.qsl[r], q = p.qsl[r + 1] - qb;
    t0 = qb + g * G;
    gcount = min(G, q - g * G);
    keys = group_keys((long long)p.seq_lens[r] - q, q, G, g, p.ratio);
  };

  // Phase B: total tiles W, the per-CTA share Q and the number of items.
  if (threadIdx.x == 0) s_max_keys = 0ull;
  __syncthreads();
  long long W = 0;
  for (int base = 0; base < total_groups; base += kPlanThreads) {
    const int gi = base + threadIdx.x;
    long long my = 0;
    if (gi < total_groups) {
      int r, t0, gc; long long keys;
      describe(gi, r, t0, gc, keys);
      my = (keys + kTileKeysPlan - 1) / kTileKeysPlan;
      if (my > 0) my += p.item_cost;
      atomicMax(&s_max_keys, (unsigned long long)keys);
    }
    long long tot;
    block_exclusive_scan(my, &tot, warp_sums);
    W += tot;
  }
  if (threadIdx.x == 0) {
    long long Q = (W + p.n_cta - 1) / p.n_cta;
    if (Q < p.min_tiles) Q = p.min_tiles;
    if (Q <= p.item_cost) Q = p.item_cost + 1;  // every used CTA keeps tiles of its own
    if (Q < 1) Q = 1;
    s_Q = Q;
    s_n_empty = 0;
  }
  __syncthreads();
  const long long Q = s_Q;
  // rows go to the workspace only when every row of the batch fits there: a
  // batch that still merges long rows inside the scoring kernel gains nothing
  // from a second kernel for the short ones
  const bool rows_ok = G == 1 && p.L.score_stride > 0 && s_max_keys <= (unsigned long long)p.L.score_stride;
  const int n_used = (int)((W + Q - 1) / Q);

  for (int i = threadIdx.x; i < kMaxCtas; i += kPlanThreads) s_wide[i] = -1;
  __syncthreads();
  // Phase C: emit the pieces in tile order; CTA c's items are contiguous.
  // Group g takes stream positions [P, P + item_cost + tiles): the charged
  // tiles first, then its own from V = P + item_cost on.
  long long tile_carry = 0, item_carry = 0, sg_carry = 0, cb_carry = 0, wide_carry = 0;
  bool overflow = false;
  for (int base = 0; base < total_groups; base += kPlanThreads) {
    const int gi = base + threadIdx.x;
    int r = 0, t0 = 0, gc = 0;
    long long keys = 0, tiles = 0, pieces = 0;
    if (gi < total_groups) {
      describe(gi, r, t0, gc, keys);
      tiles = (keys + kTileKeysPlan - 1) / kTileKeysPlan;
    }
    // a decode row short enough is scored into the workspace (no merge)
    const bool to_rows = rows_ok && keys > 0;
    if (to_rows) row_keys[t0] = (int32_t)keys;
    long long t_tiles;
    const long long cost = tiles > 0 ? tiles + p.item_cost : 0;
    const long long P = tile_carry + block_exclusive_scan(cost, &t_tiles, warp_sums);
    const long long V = P + (tiles > 0 ? p.item_cost : 0);
    if (tiles > 0) pieces = (V + tiles - 1) / Q - V / Q + 1;
    const bool is_split = pieces > 1 && !to_rows;
    long long t_items, t_sg, t_cb;
    const long long my_item = item_carry + block_exclusive_scan(pieces, &t_items, warp_sums);
    const long long my_sg = sg_carry + block_exclusive_scan(is_split ? 1 : 0, &t_sg, warp_sums);
    const long long my_cb =
        cb_carry + block_exclusive_scan(is_split ? (long long)gc * pieces : 0, &t_cb, warp_sums);
    const bool fits = my_item + pieces <= p.L.max_items &&
                      (!is_split || (my_sg < p.L.max_split_groups &&
                                     my_cb + (long long)gc * pieces <= p.L.max_cand_blocks));
    if (!fits) overflow = true;
    const bool is_wide = fits && is_split && G == 1 && pieces >= kWideSplit;
    long long t_wide;
    const long long my_wide = wide_carry + block_exclusive_scan(is_wide ? 1 : 0, &t_wide, warp_sums);
    if (is_wide && my_wide < p.L.max_wide) s_wide[my_sg] = (int32_t)my_wide;
    wide_carry += t_wide;
    for (long long j = 0; j < pieces && fits; ++j) {
      const long long c = V / Q + j;  // CTA of this piece
      const long long s0 = max(V, c * Q), s1 = min(V + tiles, (c + 1) * Q);
      Item it;
      it.r = r;
      it.t0 = t0;
      it.gcount = gc;
      it.k0 = (int)((s0 - V) * kTileKeysPlan);
      it.k1 = (int)min((s1 - V) * kTileKeysPlan, keys);
      it.split = (int)j | ((int)pieces << 16);
      it.cand_block = is_split ? (int)my_cb : -1;
      it.sgroup = to_rows ? kSgroupRows : (is_split ? (int)my_sg : -1);
      items[my_item + j] = it;
      // the piece that opens CTA c: its range starts at c * Q, or CTA c
      // starts among the tiles charged to this group
      if (s0 == c * Q || (j == 0 && c * Q >= P)) cta_start[c] = (int)(my_item + j);
    }
    tile_carry += t_tiles;
    item_carry += t_items;
    sg_carry += t_sg;
    cb_carry += t_cb;
    if (p.ratio > 1) {
      // a compressed cache leaves the first rows of a request without a visible
      // entry: no item covers them, so their rows are all -1, written here a
      // warp per group
      if (gi < total_groups && keys == 0) s_empty[atomicAdd(&s_n_empty, 1)] = make_int2(t0, gc);
      __syncthreads();
      const int n_empty = s_n_empty;
      const int lane = threadIdx.x & 31;
      for (int e = threadIdx.x >> 5; e < n_empty; e += kPlanThreads / 32) {
        const int2 ge = s_empty[e];
        for (int t = ge.x; t < ge.x + ge.y; ++t)
          for (int i = lane; i < p.index_topk; i += 32)
            p.topk_buffer[(size_t)t * p.index_topk + i] = -1;
      }
      __syncthreads();
      if (threadIdx.x == 0) s_n_empty = 0;
      __syncthreads();
    }
  }
  const int any_overflow = __syncthreads_or(overflow ? 1 : 0);
  // each split group's wide index; the shared histograms of wide groups start
  // empty (a merge empties its group's again, for the next layer of a stack)
  {
    int32_t* wide_of = reinterpret_cast<int32_t*>(p.ws + p.L.wide_of);
    const int nsg = (int)min(sg_carry, (long long)p.L.max_split_groups);
    for (int sg = threadIdx.x; sg < nsg; sg += kPlanThreads) wide_of[sg] = s_wide[sg];
    uint4* gh = reinterpret_cast<uint4*>(p.ws + p.L.ghist);
    const int n_wide = any_overflow ? 0 : (int)min(wide_carry, (long long)p.L.max_wide);
    for (int i = threadIdx.x; i < n_wide * (kSharedHistWords / 4); i += kPlanThreads)
      gh[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (any_overflow) raise_status(p.status, kStatusBadMetadata);
  if (any_overflow && p.L.score_stride > 0)
    for (int t = threadIdx.x; t < p.T; t += kPlanThreads) row_keys[t] = 0;
  const int n_items = any_overflow ? 0 : (int)item_carry;
  for (int c = threadIdx.x; c <= p.n_cta; c += kPlanThreads)
    if (any_overflow || c >= n_used) cta_start[c] = n_items;
  __syncthreads();  // every CTA's range and items are written
  CtaHead* heads = reinterpret_cast<CtaHead*>(p.ws + p.L.heads);
  for (int c = threadIdx.x; c < p.n_cta; c += kPlanThreads) {
    CtaHead h;
    h.it_begin = cta_start[c];
    h.it_end = cta_start[c + 1];
    h.first = h.it_begin < h.it_end ? items[h.it_begin] : Item{};
    h.pad[0] = h.pad[1] = 0;
    heads[c] = h;
  }
  for (int i = threadIdx.x; i < (int)min(sg_carry, (long long)p.L.max_split_groups); i += kPlanThreads)
    done[i] = 0;
  if (threadIdx.x == 0) {
    hdr->n_items = n_items;
    hdr->n_split_groups = (int32_t)sg_carry;
    hdr->n_cand_blocks = (int32_t)cb_carry;
    hdr->tiles_per_cta = (int32_t)Q;
    hdr->total_groups = total_groups;
    hdr->n_used_ctas = n_used;
  }
}

}  // namespace dsa
