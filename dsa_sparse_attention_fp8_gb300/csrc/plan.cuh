// Device-side batch plan: turns (query_start_loc, seq_lens) into the list of
// work items the scoring kernel walks, without any host round trip.
//
// A work item is (request r, a group of up to G consecutive query rows of r,
// a key range [k0, k1) of r's context).  Groups of rows share every key tile
// they load (the rows' heads are the N side of one MMA).  A group whose
// visible context is longer than the split length S is cut into key ranges
// ("splits") that run on different SMs; each split keeps an exact local
// top-k and the last split of a group to finish merges them.
//
// S = clamp(total visible keys / target items, min_split, max_split), so the
// number of items is at most (#groups + target) and at most `target` groups
// are split whenever S is not capped by max_split (the host sizes the
// workspace for the capped case too).
#pragma once

#include <cstdint>

#include "kwrite.cuh"

namespace dsa {

struct Item {
  int32_t r;           // request
  int32_t t0;          // first query row of the group
  int32_t gcount;      // rows in the group (1..G)
  int32_t k0, k1;      // key range [k0, k1) (logical positions); k0 % 128 == 0
  int32_t split;       // split index | (number of splits << 16)
  int32_t cand_block;  // first candidate block of the group (split groups), else -1
  int32_t sgroup;      // split-group id (index of its done counter), else -1
};
static_assert(sizeof(Item) == 32, "Item must stay 32 bytes");

constexpr int kMaxTarget = 320;     // upper bound on work-item target (2 per SM, <=160 SMs)
constexpr int kPlanThreads = 1024;

struct PlanHeader {
  int32_t n_items;
  int32_t n_split_groups;
  int32_t n_cand_blocks;
  int32_t split_len;
  int32_t total_groups;
  int32_t pad[59];
};
static_assert(sizeof(PlanHeader) == 256, "PlanHeader is one 256-byte line");

// Workspace carve-up; identical on host and device.
struct WsLayout {
  size_t header, group_prefix, items, done, cand_count, cand_keys, cand_idx, total;
  int max_items, max_split_groups, max_cand_blocks;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline WsLayout ws_layout(int T, int R, int G, int k) {
  WsLayout L;
  L.max_items = T + kMaxTarget;
  L.max_split_groups = kMaxTarget;
  L.max_cand_blocks = G * 2 * kMaxTarget;
  size_t o = 0;
  L.header = o;       o = align256(o + sizeof(PlanHeader));
  L.group_prefix = o; o = align256(o + sizeof(int32_t) * (size_t)(R + 1));
  L.items = o;        o = align256(o + sizeof(Item) * (size_t)L.max_items);
  L.done = o;         o = align256(o + sizeof(int32_t) * (size_t)L.max_split_groups);
  L.cand_count = o;   o = align256(o + sizeof(int32_t) * (size_t)L.max_cand_blocks);
  L.cand_keys = o;    o = align256(o + sizeof(uint32_t) * (size_t)L.max_cand_blocks * k);
  L.cand_idx = o;     o = align256(o + sizeof(int32_t) * (size_t)L.max_cand_blocks * k);
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
  int R, T, G, max_blocks, index_topk, target;
  int min_split, max_split;  // bounds on the split length S (multiples of 128)
  int32_t* topk_buffer;  // for -1 rows of malformed requests
  unsigned char* ws;
  WsLayout L;
  int32_t* status;
};

// Keys visible to the last row of group g of a request with prefix P and q new rows.
__device__ __forceinline__ long long group_keys(long long P, int q, int G, int g) {
  const int last = min((g + 1) * G, q);
  return P + last;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
  __shared__ long long warp_sums[32];
  __shared__ int s_split_len;
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(p.ws + p.L.header);
  int32_t* group_prefix = reinterpret_cast<int32_t*>(p.ws + p.L.group_prefix);
  Item* items = reinterpret_cast<Item*>(p.ws + p.L.items);
  int32_t* done = reinterpret_cast<int32_t*>(p.ws + p.L.done);
  const int G = p.G;

  // Phase A: groups per request (prefix sums) and the total number of visible keys.
  long long groups_carry = 0, keys_acc = 0;
  for (int base = 0; base < p.R; base += kPlanThreads) {
    const int r = base + threadIdx.x;
    long long groups = 0;
    if (r < p.R) {
      const int qb = p.qsl[r], qe = p.qsl[r + 1];
      const int q = qe - qb, seq = p.seq_lens[r];
      const bool bad = q < 0 || seq < q || (long long)seq > (long long)p.max_blocks * kPageTokens ||
                       qb < 0 || qe > p.T;
      if (bad) {
        raise_status(p.status, kStatusBadMetadata);
        // rows of a malformed request hold no indices
        for (int t = max(qb, 0); t < min(qe, p.T); ++t)
          for (int i = 0; i < p.index_topk; ++i) p.topk_buffer[(size_t)t * p.index_topk + i] = -1;
      } else if (q > 0) {
        groups = (q + G - 1) / G;
        const long long P = seq - q;
        const long long nfull = q / G;
        keys_acc += nfull * P + (long long)G * nfull * (nfull + 1) / 2;
        if (q % G) keys_acc += P + q;
      }
    }
    long long tot;
    const long long ex = block_exclusive_scan(groups, &tot, warp_sums);
    if (r < p.R) group_prefix[r] = (int32_t)(groups_carry + ex);
    groups_carry += tot;
  }
  {
    long long tot;
    block_exclusive_scan(keys_acc, &tot, warp_sums);
    if (threadIdx.x == 0) {
      group_prefix[p.R] = (int32_t)groups_carry;
      long long S = (tot + p.target - 1) / p.target;
      S = ((S + 127) / 128) * 128;
      if (S < p.min_split) S = p.min_split;
      if (S > p.max_split) S = p.max_split;
      if (S < 128) S = 128;
      s_split_len = (int)S;
    }
  }
  __syncthreads();
  const int total_groups = (int)groups_carry;
  const long long S = s_split_len;

  // Phase B: count items / split groups / candidate blocks (for reversed placement).
  auto describe = [&](int gi, int& r, int& t0, int& gcount, long long& keys, int& nsplit) {
    int lo = 0, hi = p.R - 1;  // last r with group_prefix[r] <= gi
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (group_prefix[mid] <= gi) lo = mid; else hi = mid - 1;
    }
    r = lo;
    const int g = gi - group_prefix[r];
    const int qb = p.qsl[r], q = p.qsl[r + 1] - qb;
    t0 = qb + g * G;
    gcount = min(G, q - g * G);
    keys = group_keys((long long)p.seq_lens[r] - q, q, G, g);
    nsplit = (int)((keys + S - 1) / S);
  };

  long long n_items = 0;
  for (int base = 0; base < total_groups; base += kPlanThreads) {
    const int gi = base + threadIdx.x;
    long long my = 0;
    if (gi < total_groups) {
      int r, t0, gc, ns; long long keys;
      describe(gi, r, t0, gc, keys, ns);
      my = ns;
    }
    long long tot;
    block_exclusive_scan(my, &tot, warp_sums);
    n_items += tot;
  }

  // Phase C: emit items, last group first (later rows of a chunk see more keys,
  // so the static round-robin over CTAs starts with the longest items).
  long long item_carry = 0, sg_carry = 0, cb_carry = 0;
  const bool overflow = n_items > p.L.max_items;
  for (int base = 0; base < total_groups; base += kPlanThreads) {
    const int gi = base + threadIdx.x;
    int r = 0, t0 = 0, gc = 0, ns = 0;
    long long keys = 0;
    if (gi < total_groups) describe(gi, r, t0, gc, keys, ns);
    const bool is_split = ns > 1;
    long long t_items, t_sg, t_cb;
    const long long ex_items = block_exclusive_scan(ns, &t_items, warp_sums);
    const long long ex_sg = block_exclusive_scan(is_split ? 1 : 0, &t_sg, warp_sums);
    const long long ex_cb = block_exclusive_scan(is_split ? (long long)gc * ns : 0, &t_cb, warp_sums);
    if (gi < total_groups && !overflow) {
      const long long my_sg = sg_carry + ex_sg;
      const long long my_cb = cb_carry + ex_cb;
      const bool fits = !is_split || (my_sg < p.L.max_split_groups &&
                                      my_cb + (long long)gc * ns <= p.L.max_cand_blocks);
      if (!fits) raise_status(p.status, kStatusBadMetadata);
      for (int j = 0; j < ns && fits; ++j) {
        Item it;
        it.r = r;
        it.t0 = t0;
        it.gcount = gc;
        it.k0 = (int)(j * S);
        it.k1 = (int)min((long long)(j + 1) * S, keys);
        it.split = j | (ns << 16);
        it.cand_block = is_split ? (int)my_cb : -1;
        it.sgroup = is_split ? (int)my_sg : -1;
        const long long slot = n_items - 1 - (item_carry + ex_items + j);
        items[slot] = it;
      }
    }
    item_carry += t_items;
    sg_carry += t_sg;
    cb_carry += t_cb;
  }
  if (overflow) raise_status(p.status, kStatusBadMetadata);
  for (int i = threadIdx.x; i < (int)min(sg_carry, (long long)p.L.max_split_groups); i += kPlanThreads)
    done[i] = 0;
  if (threadIdx.x == 0) {
    hdr->n_items = overflow ? 0 : (int32_t)n_items;
    hdr->n_split_groups = (int32_t)sg_carry;
    hdr->n_cand_blocks = (int32_t)cb_carry;
    hdr->split_len = (int32_t)S;
    hdr->total_groups = total_groups;
  }
}

}  // namespace dsa
