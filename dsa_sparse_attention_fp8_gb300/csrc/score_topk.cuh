// Paged lightning-indexer scoring + exact streaming top-k, one persistent
// kernel per F layer.
//
// Score (DeepSeek-V3.2 report, arXiv:2512.02556, listed in the references of
// "GLM-5.3 推理全链路(十二)"):
//   score(t, s) = k_scale[s] * sum_h (w[t,h] * q_scale[t,h]) * ReLU(q[t,h] . k[s])
// with q, k the E4M3 codes; the FP32 scales are positive, so they factor out
// of the ReLU.  Keys are gathered page by page through the block table
// ("GLM-5.3 推理全链路(十二)", "64 token 页的由来": the paged-MQA read is by
// 64-token pages); the result is the top `index_topk` key positions per query
// row, -1 padded ("vLLM IndexCache 实战指南" §二: -1 clear, then scatter into
// the shared [max_num_batched_tokens, index_topk] buffer).
//
// Structure (one CTA per SM, 10 warps):
//   warp 0      producer: per page of a key tile (128 keys = 2 pages, or 4
//               pages for the 256-key decode stages) one TMA load of its
//               64 x 128 B key rows into a 128B-swizzled stage and one of its
//               256 B of scales into a ring of scale slots, both counted by
//               one expect-tx arrival; the query tile of each item
//               (double-buffered when it is small).
//   warp 1      owns tensor memory; one lane issues 4 tcgen05.mma (K = 32
//               each) per 128-key block: D[key, row*H + head] += k . q, FP32
//               in TMEM.
//   warps 2-9   epilogue, two warpgroups; thread = one key row of the tile
//               (its TMEM lane).  Each warpgroup takes two of its blocks per
//               iteration: for each query row of the group it reads the H
//               accumulators of both, ReLU, weight and sum them in two
//               interleaved chains, times the keys' scales, then streams the
//               scores into an exact top-k buffer in shared memory (append
//               above the running threshold; when the buffer nears full,
//               select in place the candidates at or above the k-th largest's
//               bin and raise the threshold).
// No score row goes to global memory (except the optional debug dump).
#pragma once

#include <cstdint>

#include "plan.cuh"
#include "ptx.cuh"

namespace dsa {

constexpr int kScoreThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kTileKeys = 128;
constexpr int kStageBytes = kTileKeys * kHeadDim;  // 16 KB of key rows
constexpr int kScaleSlotBytes = kTileKeys * 4;      // the FP32 scales of one tile's keys
constexpr int kMaxStages = 16;
constexpr int kMaxAccBufs = 8;
constexpr int kMaxQBufs = 2;
constexpr int kTmemCols = 512;

struct TokSlot {
  int32_t count;   // candidates held
  uint32_t thr;    // keys <= thr are not admitted
  int32_t pos;     // last cache entry the query row sees (its position when uncompressed)
  int32_t t;       // query row
};

struct ScoreParams {
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int max_blocks;
  const uint8_t* k_cache;
  int64_t num_pages;
  const float* q_scale;
  const float* w;
  int T, H, G, k, C, NS, NB, NQ, NR, n_max;
  int lg_nb, lg_nr;  // NB = 1 << lg_nb accumulator buffers, NR = 1 << lg_nr scale slots
  int BPS;           // 128-key MMA blocks per pipeline stage (1 or 2); a tile = one stage
  int lg_bps;        // BPS = 1 << lg_bps
  int ratio;         // tokens per cache entry: a row at pos sees entries < (pos + 1) / ratio
  int q_box_per_token;
  // 1 when the kernel that precedes this one in the stream is this layer's
  // cache write, launched after the plan completed: the plan's outputs (items,
  // cta_start) and every cache entry below a request's first new entry may
  // then be read before the programmatic-launch wait, overlapping the write
  int meta_ready;
  // 1 when q_fp8 is not written by the preceding kernel (may be loaded before the wait)
  int q_ready;
  uint32_t q_bytes;  // bytes of one query-tile buffer
  const Item* items;
  const int32_t* cta_start;  // CTA c walks items [cta_start[c], cta_start[c+1])
  const CtaHead* heads;      // per CTA: that range and its first item
  int CB;                    // capacity of one candidate block
  uint32_t* cand_keys;
  int32_t* cand_idx;
  uint16_t* cand_hist;   // per candidate block: level-1 histogram (kBlockBins; counts <= CB)
  uint16_t* cand_start;  // per candidate block: start offset of every bin
  int32_t* cand_count;
  uint32_t* ghist;       // per wide split group: the pieces' shared histograms
                         // (early-bound level-1 bins, then final-candidate level-1 bins)
  const int32_t* wide_of;  // per split group: its wide index, or -1
  int32_t* done;
  int32_t* topk;
  float* scores_out;
  int64_t scores_ld;
  uint32_t* score_rows;      // [T, score_stride] keys of rows scored into the workspace
  int score_stride;
  int32_t* status;
  // iterations a wait on another role may take before it gives up (kWaitLimit
  // unless lowered to test the timeout path)
  uint32_t wait_limit;
  // dynamic shared memory offsets (from a 1024-aligned base)
  uint32_t off_stage, off_scale, off_q, off_ckeys, off_cidx, off_wq, off_tok, off_hist, off_misc,
      off_bar;
};

struct SelScratch {
  int scan[16];                // per-warp partials of a scan (up to 256 threads), 2 buffers
  int res[4];                  // a bin search's result (bin, above, count)
  uint32_t table[256];         // sub-bin counts while a cut bin is refined
};

struct Misc {
  int abort;       // any role gave up (producer and MMA stop early on it)
  uint32_t tmem_base;
  int merge_flag;
  int epi_abort;   // an epilogue wait gave up; read by the epilogue only after barriers
  SelScratch sel[2];
  int2 piece_pre[2 * (kMaxCtas + 1)];  // per selector: a merge's piece prefix sums
};

// The candidates of one query row are selected by a "selector": either one
// warpgroup (128 threads, its own rows) or both (256 threads, the single row
// of a decode item).  A selector names its threads, its named barrier and its
// scratch.
//
// Selection runs once per row and item, so its code is written as small
// rolled loops in out-of-line functions: a long unrolled sequence that runs
// once costs an instruction-cache miss per 128 bytes of code, which on this
// part dominated the arithmetic.  Candidates stay in shared memory (key
// buffer ck, index buffer ci; key 0 = none) and are visited as chunks of nt:
// candidate i = chunk * nt + tid.
struct Selector {
  int nt;          // threads
  int tid;         // this thread, 0..nt-1
  uint32_t bar;    // named barrier id
  int* unused;
  SelScratch* s;
};

constexpr int kBins = 2048;
constexpr int kHistShift = 21;  // level-1 bin of a key: its top 11 bits (sign, exponent, 2 mantissa)

struct Thresh {
  uint32_t prefix;  // keys >= prefix are taken (early), or > prefix plus `need` ties (exact)
  int need;
  int early;
};

struct BinCut {
  int bin;    // the bin holding the need-th largest key
  int above;  // keys in higher bins
  int cnt;    // keys in that bin
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint32_t warp_inclusive_sum(uint32_t x) {
  const int lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__device__ __forceinline__ uint32_t u4_at(const uint4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

__device__ __forceinline__ void clear_bins(const Selector S, uint32_t a, int nbins) {
  for (int b = 4 * S.tid; b < nbins; b += 4 * S.nt) sts_v4(a + 4u * b, make_uint4(0, 0, 0, 0));
}

// Exclusive scan of one value per selector thread (one barrier); *total gets
// the sum.  Scratch buffer `buf` (0/1) is reused only after another barrier
// of the selector.
__device__ __forceinline__ uint32_t sel_scan(const Selector S, uint32_t v, uint32_t* total,
                                             int buf = 0) {
  const int lane = S.tid & 31, w = S.tid >> 5, nw = S.nt >> 5;
  int* sc = S.s->scan + 8 * buf;
  const uint32_t inc = warp_inclusive_sum(v);
  if (lane == 31) sc[w] = (int)inc;
  named_bar_sync(S.bar, S.nt);
  uint32_t off = inc - v, tot = 0;
  for (int u = 0; u < nw; ++u) {
    const uint32_t c = (uint32_t)sc[u];
    off += u < w ? c : 0u;
    tot += c;
  }
  *total = tot;
  return off;
}

// In an nbins-bin histogram (shared memory; nbins/nt in {4, 8, 16}), the bin
// where the count from the top reaches `need` (1 <= need <= total).  Thread t
// holds the nbins/nt consecutive bins below the top t*nbins/nt in registers; a
// scan over threads finds the owner of the crossing, which walks its bins.
__device__ __noinline__ BinCut find_bin(const Selector S, uint32_t hist_s, int nbins, int need) {
  const int per = nbins / S.nt;
  const uint32_t lo = (uint32_t)(nbins - (S.tid + 1) * per);  // this thread's lowest bin
  uint4 q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = 4 * i < per ? lds_v4(hist_s + 4u * (lo + 4u * i)) : make_uint4(0, 0, 0, 0);
  uint32_t local = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) local += q[i].x + q[i].y + q[i].z + q[i].w;
  uint32_t tot;
  uint32_t above = sel_scan(S, local, &tot);  // threads before this one hold higher bins
  const uint32_t un = (uint32_t)need;
  if (above < un && un <= above + local) {
    int bin = (int)lo + per - 1;
    uint32_t cnt = 0;
#pragma unroll
    for (int i = 15; i >= 0; --i) {  // from this thread's highest bin down
      if (i < per) {
        const uint32_t c = u4_at(q[i >> 2], i & 3);
        if (cnt == 0 && un <= above + c) {
          bin = (int)lo + i;
          cnt = c;
        } else if (cnt == 0) {
          above += c;
        }
      }
    }
    S.s->res[0] = bin;
    S.s->res[1] = (int)above;
    S.s->res[2] = (int)cnt;
  }
  named_bar_sync(S.bar, S.nt);
  const BinCut r{S.s->res[0], S.s->res[1], S.s->res[2]};
  named_bar_sync(S.bar, S.nt);  // result read before the scratch is reused
  return r;
}

// find_bin over a histogram of nbins bins in global memory (read from L2:
// other SMs add to it; nbins / S.nt a multiple of 4); the bin is -1 when the
// histogram holds fewer than `need` keys.
__device__ __noinline__ BinCut find_bin_global(const Selector S, const uint32_t* hist, int nbins,
                                               int need) {
  const int per = nbins / S.nt;
  const int nq = per / 4;  // this thread's bins as uint4 words
  const uint32_t lo = (uint32_t)(nbins - (S.tid + 1) * per);
  const uint4* h4 = reinterpret_cast<const uint4*>(hist + lo);
  uint32_t local = 0;
  for (int i = 0; i < nq; i += 4) {
    uint4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) q[u] = i + u < nq ? __ldcg(h4 + i + u) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u) local += q[u].x + q[u].y + q[u].z + q[u].w;
  }
  uint32_t tot;
  uint32_t above = sel_scan(S, local, &tot);
  const uint32_t un = (uint32_t)need;
  if (S.tid == 0 && tot < un) S.s->res[0] = -1;
  if (tot >= un && above < un && un <= above + local) {
    // walk this thread's bins from the top, 16 at a time
    for (int c = (nq + 3) / 4 - 1; c >= 0; --c) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        q[u] = 4 * c + u < nq ? __ldcg(h4 + 4 * c + u) : make_uint4(0, 0, 0, 0);
      bool found = false;
#pragma unroll
      for (int i = 15; i >= 0; --i) {
        const uint32_t cnt = u4_at(q[i >> 2], i & 3);
        if (16 * c + i < per && !found && un <= above + cnt) {
          S.s->res[0] = (int)lo + 16 * c + i;
          S.s->res[1] = (int)above;
          S.s->res[2] = (int)cnt;
          found = true;
        } else if (!found) {
          above += cnt;
        }
      }
      if (found) break;
    }
  }
  named_bar_sync(S.bar, S.nt);
  const BinCut r{S.s->res[0], S.s->res[1], S.s->res[2]};
  named_bar_sync(S.bar, S.nt);
  return r;
}

__device__ __forceinline__ bool sel_above(uint32_t key, Thresh th) {
  return key != 0u && (th.early ? key >= th.prefix : key > th.prefix);
}
__device__ __forceinline__ bool sel_tie(uint32_t key, Thresh th) {
  return key != 0u && !th.early && key == th.prefix;
}

// Selection passes visit the slot's candidates in batches of kSelBatch per
// thread (candidate i = (b * kSelBatch + u) * nt + tid): a rolled loop whose
// body loads a whole batch before using it.  One-shot code that is unrolled
// further runs at the instruction-fetch rate on this part, so the passes are
// kept small and re-read shared memory instead of holding candidates in
// registers.
constexpr int kSelBatch = 8;

// Warp-level search of a small histogram (nbins = 256 or 32, shared memory)
// from the top for the bin where the running count reaches `need` (1 <= need
// <= total): lane l sums the nbins/32 bins below the top l*nbins/32, a warp
// scan finds the crossing lane, which walks its bins.  Every calling warp
// computes the same answer, so no barrier is needed to share it.
__device__ __forceinline__ BinCut find_bin_warp(uint32_t hist_s, int nbins, int need) {
  const int lane = lane_id();
  const int per = nbins >> 5;  // 8 or 1
  const uint32_t lo = (uint32_t)(nbins - (lane + 1) * per);
  uint32_t h[8];
  if (per == 8) {
    const uint4 a = lds_v4(hist_s + 4u * lo), b = lds_v4(hist_s + 4u * (lo + 4u));
    h[0] = a.x; h[1] = a.y; h[2] = a.z; h[3] = a.w; h[4] = b.x; h[5] = b.y; h[6] = b.z; h[7] = b.w;
  } else {
    h[0] = lds_u32(hist_s + 4u * lo);
#pragma unroll
    for (int i = 1; i < 8; ++i) h[i] = 0u;
  }
  uint32_t local = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) local += h[i];
  const uint32_t inc = warp_inclusive_sum(local);
  const uint32_t un = (uint32_t)need;
  const int L = __ffs(__ballot_sync(0xffffffffu, inc - local < un && un <= inc)) - 1;
  uint32_t above = inc - local, bin = lo, cnt = 0;
  bool found = false;
#pragma unroll
  for (int i = 7; i >= 0; --i) {
    const bool here = !found && i < per && un <= above + h[i];
    bin = here ? lo + (uint32_t)i : bin;
    cnt = here ? h[i] : cnt;
    above += (!found && !here && i < per) ? h[i] : 0u;
    found = found || here;
  }
  BinCut r;
  r.bin = (int)__shfl_sync(0xffffffffu, bin, L);
  r.above = (int)__shfl_sync(0xffffffffu, above, L);
  r.cnt = (int)__shfl_sync(0xffffffffu, cnt, L);
  return r;
}

// Exact threshold of the k-th largest of the slot's n keys, starting from the
// level-1 bin cut `c`: refine inside that bin on key bits 20..13, 12..5 and
// 4..0 (histograms of 256, 256 and 32 bins in scratch_s, each searched by
// every warp on its own).  Stops as soon as a whole sub-bin is taken.  The
// caller's reads of scratch_s are complete.
__device__ __noinline__ Thresh refine_in_bin(const Selector S, uint32_t ck_s, int n, BinCut c,
                                             int k, uint32_t scratch_s, int coarse_limit = 0) {
  Thresh th{(uint32_t)c.bin << kHistShift, k - c.above, 0};
  uint32_t mask = 0xFFFFFFFFu << kHistShift;
  if (c.cnt == th.need) {
    th.early = 1;
    return th;
  }
  for (int level = 0; level < 3; ++level) {
    const int shift = level == 0 ? 13 : (level == 1 ? 5 : 0);
    const int nb = level == 2 ? 32 : 256;
    const uint32_t dm = (uint32_t)nb - 1u;
    for (int b = S.tid; b < nb; b += S.nt) sts_u32(scratch_s + 4u * (uint32_t)b, 0u);
    named_bar_sync(S.bar, S.nt);
    for (int i0 = S.tid; i0 < n; i0 += kSelBatch * S.nt) {
      uint32_t kk[kSelBatch];
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        const int i = i0 + u * S.nt;
        kk[u] = lds_u32_if(i < n, ck_s + 4u * (uint32_t)i);
      }
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u)
        red_add_shared_if(kk[u] != 0u && (kk[u] & mask) == th.prefix,
                          scratch_s + 4u * ((kk[u] >> shift) & dm), 1u);
    }
    named_bar_sync(S.bar, S.nt);
    const BinCut c2 = find_bin_warp(scratch_s, nb, th.need);
    if (level == 0 && c.above + c2.above + c2.cnt <= coarse_limit) {
      // keep the whole sub-bin of the k-th largest: a superset within the limit
      th.prefix |= (uint32_t)c2.bin << shift;
      th.early = 1;
      break;
    }
    th.need -= c2.above;
    th.prefix |= (uint32_t)c2.bin << shift;
    mask |= dm << shift;
    if (c2.cnt == th.need) {
      th.early = 1;
      break;
    }
    named_bar_sync(S.bar, S.nt);  // every warp has read the scratch before it is cleared
  }
  return th;
}

constexpr int kCompactGroups = 8;  // 32-candidate groups per warp and batch
constexpr int kMergeUnits = 8;     // 32-candidate units per warp and batch of a merge's gather

// In-place compaction of a slot's n candidates to those with key >= lo
// (an early threshold: no ties to ration); returns how many are kept.
// Batches of kCompactGroups groups of 32 consecutive candidates per warp: a
// group's kept ones go out in lane order after those of the warp's earlier
// groups, of the lower warps and of earlier batches, so every write lands at
// or below the candidates still to be read; one barrier per batch exchanges
// the warps' counts once every thread holds its batch.
__device__ __noinline__ int compact_early(const Selector S, int n, uint32_t ck_s, uint32_t ci_s,
                                          uint32_t lo) {
  const int lane = S.tid & 31, w = S.tid >> 5, nw = S.nt >> 5;
  const uint32_t lt = lanemask_lt();
  if (lo == 0u) lo = 1u;  // key 0 never enters a slot
  const int per_batch = kCompactGroups * S.nt;
  int carry = 0;
  for (int b0 = 0, it = 0; b0 < n; b0 += per_batch, ++it) {
    const int i0 = b0 + w * (kCompactGroups * 32) + lane;
    uint32_t kk[kCompactGroups], ix[kCompactGroups], m[kCompactGroups];
#pragma unroll
    for (int u = 0; u < kCompactGroups; ++u) kk[u] = lds_u32_if(i0 + 32 * u < n, ck_s + 4u * (uint32_t)(i0 + 32 * u));
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kCompactGroups; ++u) {
      m[u] = __ballot_sync(0xffffffffu, kk[u] >= lo);
      cnt += __popc(m[u]);
    }
    int* buf = S.s->scan + 8 * (it & 1);
    if (lane == 0) buf[w] = cnt;
#pragma unroll
    for (int u = 0; u < kCompactGroups; ++u)
      ix[u] = lds_u32_if((m[u] >> lane) & 1u, ci_s + 4u * (uint32_t)(i0 + 32 * u));
    named_bar_sync(S.bar, S.nt);
    int a = carry, tot = 0;
    for (int v = 0; v < nw; ++v) {
      const int c = buf[v];
      a += v < w ? c : 0;
      tot += c;
    }
#pragma unroll
    for (int u = 0; u < kCompactGroups; ++u) {
      const uint32_t pos = (uint32_t)(a + __popc(m[u] & lt));
      const bool wr = (m[u] >> lane) & 1u;
      sts_u32_if(wr, ck_s + 4u * pos, kk[u]);
      sts_u32_if(wr, ci_s + 4u * pos, ix[u]);
      a += __popc(m[u]);
    }
    carry += tot;
  }
  return carry;
}

enum SelMode {
  kSelRow = 0,     // exact top-min(n, k) indices to a row of the top-k buffer, -1 after
  kSelBlock = 1,   // a superset of the top-k of at most `limit` to a candidate block
  kSelInPlace = 2  // the same superset kept in the slot; histogram and threshold follow
};

// One selection over a slot's n candidates (key buffer ck_s, index buffer
// ci_s, level-1 histogram hist_s).  kSelBlock / kSelInPlace keep every
// candidate if n <= limit, else every one in or above the level-1 bin of the
// k-th largest if that fits, else exactly k.  Output order is the buffer's
// order (deterministic); ties at an exact threshold are taken in that order
// up to the quota.  `known`, if given, is the level-1 cut of the k-th largest
// (hist_s is then only scratch).  Row output is staged in shared memory
// (hist_s, after its last use) and copied out coalesced; in place, the kept
// candidates are held in registers one batch at a time behind a barrier per
// batch (an early threshold goes to compact_early), and the histogram is
// updated without recounting.  Returns the number written; for kSelInPlace
// *thr gets the admission threshold of the kept set.
__device__ __noinline__ int slot_select(const Selector S, int mode, int n, uint32_t ck_s,
                                        uint32_t ci_s, uint32_t hist_s, int k, int limit,
                                        uint32_t* gk, int32_t* gi, uint32_t* thr,
                                        const BinCut* known = nullptr,
                                        const Thresh* given = nullptr) {
  if (mode == kSelRow && n <= k) {
    for (int i = S.tid; i < k; i += S.nt)
      __stcg(gi + i, i < n ? (int32_t)lds_u32(ci_s + 4u * (uint32_t)i) : -1);
    return n;
  }
  if (mode != kSelRow && n <= limit) {
    if (mode == kSelBlock)
      for (int i = S.tid; i < n; i += S.nt) {
        __stcg(gk + i, lds_u32(ck_s + 4u * (uint32_t)i));
        __stcg(gi + i, (int32_t)lds_u32(ci_s + 4u * (uint32_t)i));
      }
    return n;
  }
  Thresh th;
  int above_cut = 0;  // candidates in the bins above the cut bin
  if (given) {
    th = *given;  // the caller's threshold (in place: keep the keys it takes)
  } else {
    // the level-1 cut, found in the histogram unless the caller knows it
    const BinCut c = known ? *known : find_bin(S, hist_s, kBins, k);
    // in place, a kept set near the limit would leave little room and bring
    // the next shrink soon: keep the whole cut bin only while it frees at
    // least half the room above k, else cut at the k-th's sub-bin (one more
    // pass), else exactly
    const int keep = mode == kSelInPlace ? k + (limit - k) / 2 : limit;
    above_cut = c.above;
    if (mode != kSelRow && c.above + c.cnt <= keep)
      th = Thresh{(uint32_t)c.bin << kHistShift, 0, 1};
    else
      th = refine_in_bin(S, ck_s, n, c, k, smem_u32(S.s->table), mode == kSelInPlace ? keep : 0);
  }
  const uint32_t quota = th.early ? 0u : (uint32_t)th.need;
  const bool in_place = mode == kSelInPlace;
  // Batch-major output order: batch b's candidates follow every kept one of
  // earlier batches, so in place a batch's writes land at or below its own
  // candidates; once every thread holds the batch it may be overwritten.
  // Inside a batch, warp w holds kSelBatch groups of 32 consecutive
  // candidates; a group's kept ones go out in lane order after those of the
  // warp's earlier groups and of the lower warps (counts from ballots, one
  // barrier to exchange the warps' totals).  An early threshold has no ties.
  uint32_t carry_a = 0, carry_t = 0;  // kept-above / tie counts of earlier batches
  if (in_place && th.early) {
    carry_a = (uint32_t)compact_early(S, n, ck_s, ci_s, th.prefix);
  } else {
    const int lane = S.tid & 31, w = S.tid >> 5, nw = S.nt >> 5;
    const uint32_t lt = lanemask_lt();
    const int per_batch = kSelBatch * S.nt;
    const bool ties = !th.early;
    for (int b0 = 0, it = 0; b0 < n; b0 += per_batch, ++it) {
      const int i0 = b0 + w * (kSelBatch * 32) + lane;
      uint32_t kk[kSelBatch], ix[kSelBatch], am[kSelBatch], tm[kSelBatch];
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        const int i = i0 + 32 * u;
        kk[u] = lds_u32_if(i < n, ck_s + 4u * (uint32_t)i);
      }
      uint32_t cnt = 0;  // this warp's above | ties << 16
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        am[u] = __ballot_sync(0xffffffffu, sel_above(kk[u], th));
        tm[u] = ties ? __ballot_sync(0xffffffffu, sel_tie(kk[u], th)) : 0u;
        cnt += (uint32_t)__popc(am[u]) + ((uint32_t)__popc(tm[u]) << 16);
      }
      int* buf = S.s->scan + 8 * (it & 1);
      if (lane == 0) buf[w] = (int)cnt;
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u)
        ix[u] = lds_u32_if(((am[u] | tm[u]) >> lane) & 1u, ci_s + 4u * (uint32_t)(i0 + 32 * u));
      named_bar_sync(S.bar, S.nt);  // the warps' totals; every thread holds its batch
      uint32_t a = carry_a, t = carry_t, tot = 0;
      for (int v = 0; v < nw; ++v) {
        const uint32_t c = (uint32_t)buf[v];
        if (v < w) {
          a += c & 0xFFFFu;
          t += c >> 16;
        }
        tot += c;
      }
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        const bool above = (am[u] >> lane) & 1u, tie = (tm[u] >> lane) & 1u;
        const uint32_t ta = t + (uint32_t)__popc(tm[u] & lt);
        const bool wr = above || (tie && ta < quota);
        const uint32_t pos = a + (uint32_t)__popc(am[u] & lt) + min(quota, ta);
        if (mode == kSelRow) {
          sts_u32_if(wr, hist_s + 4u * pos, ix[u]);
        } else if (mode == kSelBlock) {
          if (wr) {
            __stcg(gk + pos, kk[u]);
            __stcg(gi + pos, (int32_t)ix[u]);
          }
        } else {
          sts_u32_if(wr, ck_s + 4u * pos, kk[u]);
          sts_u32_if(wr, ci_s + 4u * pos, ix[u]);
        }
        a += (uint32_t)__popc(am[u]);
        t += (uint32_t)__popc(tm[u]);
      }
      carry_a += tot & 0xFFFFu;
      carry_t += tot >> 16;
    }
  }
  const int total = (int)(carry_a + min(quota, carry_t));
  named_bar_sync(S.bar, S.nt);
  if (mode == kSelRow) {
    for (int i = S.tid; i < k; i += S.nt)
      __stcg(gi + i, i < total ? (int32_t)lds_u32(hist_s + 4u * (uint32_t)i) : -1);
  } else if (in_place) {
    *thr = th.early ? (th.prefix > 0u ? th.prefix - 1u : 0u) : th.prefix;
    // The kept set's histogram without recounting: every candidate of the
    // bins above the cut bin is kept, none below it; the cut bin keeps its
    // count when the threshold is its lower edge, else the rest of `total`.
    const uint32_t cb = th.prefix >> kHistShift;
    const bool whole = th.early && (th.prefix & ((1u << kHistShift) - 1u)) == 0u;
    for (uint32_t b = (uint32_t)S.tid; b <= cb; b += (uint32_t)S.nt)
      if (b < cb || !whole) sts_u32(hist_s + 4u * b, b < cb ? 0u : (uint32_t)(total - above_cut));
    named_bar_sync(S.bar, S.nt);
  }
  return total;
}

// One pass over a slot's n candidates: every one with key >= hi goes to the
// row gi (in the slot's order; places at or beyond gi_cap, which a consistent
// histogram never yields, are not written), every one in [lo, hi) to the
// front of the slot (in place), the rest are dropped.  Returns the two counts
// (x: sent to the row, y: kept in the slot); the slot is consistent after the
// call.
// Batches of kCompactGroups groups of 32 consecutive candidates per warp,
// counts by ballots, one barrier per batch as in compact_early.
__device__ __noinline__ int2 split_pass(const Selector S, int n, uint32_t ck_s, uint32_t ci_s,
                                        uint32_t lo, uint64_t hi, int32_t* gi, int gi_cap) {
  const int lane = S.tid & 31, w = S.tid >> 5, nw = S.nt >> 5;
  const uint32_t lt = lanemask_lt();
  const int per_batch = kCompactGroups * S.nt;
  int carry_a = 0, carry_c = 0;
  for (int b0 = 0, it = 0; b0 < n; b0 += per_batch, ++it) {
    const int i0 = b0 + w * (kCompactGroups * 32) + lane;
    uint32_t kk[kCompactGroups], ix[kCompactGroups], ma[kCompactGroups], mc[kCompactGroups];
#pragma unroll
    for (int u = 0; u < kCompactGroups; ++u)
      kk[u] = lds_u32_if(i0 + 32 * u < n, ck_s + 4u * (uint32_t)(i0 + 32 * u));
    uint32_t cnt = 0;  // this warp's above | cut << 16
#pragma unroll
    for (int u = 0; u < kCompactGroups; ++u) {
      const bool above = (uint64_t)kk[u] >= hi;
      ma[u] = __ballot_sync(0xffffffffu, above);
      mc[u] = __ballot_sync(0xffffffffu, !above && kk[u] != 0u && kk[u] >= lo);
      cnt += (uint32_t)__popc(ma[u]) + ((uint32_t)__popc(mc[u]) << 16);
    }
    int* buf = S.s->scan + 8 * (it & 1);
    if (lane == 0) buf[w] = (int)cnt;
#pragma unroll
    for (int u = 0; u < kCompactGroups; ++u)
      ix[u] = lds_u32_if(((ma[u] | mc[u]) >> lane) & 1u, ci_s + 4u * (uint32_t)(i0 + 32 * u));
    named_bar_sync(S.bar, S.nt);  // the warps' counts; every thread holds its batch
    int a = carry_a, cc = carry_c;
    uint32_t tot = 0;
    for (int v = 0; v < nw; ++v) {
      const uint32_t x = (uint32_t)buf[v];
      if (v < w) {
        a += (int)(x & 0xFFFFu);
        cc += (int)(x >> 16);
      }
      tot += x;
    }
#pragma unroll
    for (int u = 0; u < kCompactGroups; ++u) {
      const int pa = a + __popc(ma[u] & lt);
      if (((ma[u] >> lane) & 1u) && pa < gi_cap) __stcg(gi + pa, (int32_t)ix[u]);
      const uint32_t pos = (uint32_t)(cc + __popc(mc[u] & lt));
      const bool wc = (mc[u] >> lane) & 1u;
      sts_u32_if(wc, ck_s + 4u * pos, kk[u]);
      sts_u32_if(wc, ci_s + 4u * pos, ix[u]);
      a += __popc(ma[u]);
      cc += __popc(mc[u]);
    }
    carry_a += (int)(tot & 0xFFFFu);
    carry_c += (int)(tot >> 16);
  }
  named_bar_sync(S.bar, S.nt);  // the kept candidates are in place
  return make_int2(carry_a, carry_c);
}

// Exact top-`need` of m <= S.nt candidates at the front of a slot to
// gi[0, need) (need <= m): thread t ranks candidate t against all m (ties by
// slot position); the ranks are distinct, so each selected candidate goes to
// its rank's position.
__device__ __forceinline__ void rank_small(const Selector S, int m, uint32_t ck_s, uint32_t ci_s,
                                           int need, int32_t* gi) {
  if (S.tid < m) {
    const uint32_t key = lds_u32(ck_s + 4u * (uint32_t)S.tid);
    int rank = 0;
    for (int j = 0; j < m; ++j) {
      const uint32_t kj = lds_u32(ck_s + 4u * (uint32_t)j);
      rank += (kj > key || (kj == key && j < S.tid)) ? 1 : 0;
    }
    if (rank < need) __stcg(gi + rank, (int32_t)lds_u32(ci_s + 4u * (uint32_t)S.tid));
  }
}

// Exact top-k of a slot's n candidates to the row gi (-1 after the last):
// one pass sends every candidate of the bins above the k-th largest's
// level-1 bin straight to the row and moves that bin's candidates to the
// front of the slot; the exact selection then runs over those alone.
__device__ __noinline__ void select_row(const Selector S, int n, uint32_t ck_s, uint32_t ci_s,
                                        uint32_t hist_s, int k, int32_t* gi) {
  if (n <= k) {
    slot_select(S, kSelRow, n, ck_s, ci_s, hist_s, k, 0, nullptr, gi, nullptr);
    return;
  }
  const BinCut c = find_bin(S, hist_s, kBins, k);
  const uint32_t lo = (uint32_t)c.bin << kHistShift;
  const int2 r = split_pass(S, n, ck_s, ci_s, lo, (uint64_t)lo + (1ull << kHistShift), gi, k);
  // r.x == c.above and r.y == c.cnt (the histogram counts the slot)
  const int above = min(r.x, k), rest = k - above;
  if (rest <= 0) return;
  if (r.y <= S.nt) {
    rank_small(S, r.y, ck_s, ci_s, rest, gi + above);
  } else {
    const BinCut cut{c.bin, 0, r.y};
    slot_select(S, kSelRow, r.y, ck_s, ci_s, hist_s, rest, 0, nullptr, gi + above, nullptr, &cut);
  }
}

// Append one candidate per thread of a warp if its key beats the threshold,
// and count it in the slot's level-1 histogram.
__device__ __forceinline__ void slot_append(uint32_t key, int32_t idx, uint32_t thr, TokSlot* ts,
                                            uint32_t* ckeys, int32_t* cidx, uint32_t hist_s) {
  const bool pass = key > thr;
  const uint32_t m = __ballot_sync(0xffffffffu, pass);
  if (m == 0) return;
  int base = 0;
  if (lane_id() == 0) base = (int)atom_add_shared(smem_u32(&ts->count), (uint32_t)__popc(m));
  base = __shfl_sync(0xffffffffu, base, 0);
  red_add_shared_if(pass, hist_s + 4 * (key >> kHistShift), 1u);
  if (pass) {
    const int p = base + __popc(m & lanemask_lt());
    ckeys[p] = key;
    cidx[p] = idx;
  }
}

// The same for two candidates per thread (two blocks of keys): one shared
// atomic reserves the warp's slots for both.
__device__ __forceinline__ void slot_append2(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib,
                                             uint32_t thr, TokSlot* ts, uint32_t* ckeys,
                                             int32_t* cidx, uint32_t hist_s) {
  const bool pa = ka > thr, pb = kb > thr;
  const uint32_t ma = __ballot_sync(0xffffffffu, pa), mb = __ballot_sync(0xffffffffu, pb);
  if ((ma | mb) == 0) return;
  const uint32_t na = (uint32_t)__popc(ma);
  int base = 0;
  if (lane_id() == 0) base = (int)atom_add_shared(smem_u32(&ts->count), na + (uint32_t)__popc(mb));
  base = __shfl_sync(0xffffffffu, base, 0);
  red_add_shared_if(pa, hist_s + 4 * (ka >> kHistShift), 1u);
  red_add_shared_if(pb, hist_s + 4 * (kb >> kHistShift), 1u);
  const uint32_t lt = lanemask_lt();
  if (pa) {
    const int q = base + __popc(ma & lt);
    ckeys[q] = ka;
    cidx[q] = ia;
  }
  if (pb) {
    const int q = base + (int)na + __popc(mb & lt);
    ckeys[q] = kb;
    cidx[q] = ib;
  }
}

// ---------------------------------------------------------------------------
// Pieces and their merge.  A piece of a split group writes, per row, a
// candidate block: its candidates (keys, indices) sorted by level-1 bin from
// the top, the block's level-1 histogram and each bin's start offset.  The
// merger finds the bin of the row's k-th largest key from the pieces'
// histograms, copies every candidate of the higher bins straight to the
// output row (they are a prefix of every block), and selects exactly among
// the candidates of that one bin.
// ---------------------------------------------------------------------------

// Publish a slot's n candidates as a bin-sorted block: histogram to ghist,
// start offsets to gstart, candidates to gk/gi.  Positions inside a bin come
// from shared atomics, so the order within a bin varies; the merger never
// depends on it except to break exact ties.  The slot's histogram becomes
// the bins' end offsets.
__device__ __forceinline__ uint2 pack16(uint4 v) {
  return make_uint2(v.x | (v.y << 16), v.z | (v.w << 16));
}

__device__ __noinline__ void slot_emit_sorted(const Selector S, int n, uint32_t ck_s, uint32_t ci_s,
                                              uint32_t hist_s, uint32_t* gk, int32_t* gi,
                                              uint16_t* ghist, uint16_t* gstart,
                                              uint32_t* shared_hist = nullptr) {
  const int per = kBins / S.nt;  // 8 or 16 consecutive bins per thread, the top first
  const uint32_t lo = (uint32_t)(kBins - (S.tid + 1) * per);
  uint4 q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    q[i] = 4 * i < per ? lds_v4(hist_s + 4u * (lo + 4u * i)) : make_uint4(0, 0, 0, 0);
  uint32_t local = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (4 * i < per) __stcg(reinterpret_cast<uint2*>(ghist + lo + 4 * i), pack16(q[i]));
    local += q[i].x + q[i].y + q[i].z + q[i].w;
  }
  if (shared_hist) {  // the group's summed histogram, for its merge
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t c = i < per ? u4_at(q[i >> 2], i & 3) : 0u;
      if (c) atomicAdd(shared_hist + lo + i, c);
    }
  }
  uint32_t tot;
  uint32_t run = sel_scan(S, local, &tot);  // candidates in higher bins; every bin is read
  uint4 st[4];
#pragma unroll
  for (int i = 3; i >= 0; --i) {
    if (4 * i < per) {
      st[i].w = run; run += q[i].w;
      st[i].z = run; run += q[i].z;
      st[i].y = run; run += q[i].y;
      st[i].x = run; run += q[i].x;
      sts_v4(hist_s + 4u * (lo + 4u * i), st[i]);
      __stcg(reinterpret_cast<uint2*>(gstart + lo + 4 * i), pack16(st[i]));
    }
  }
  named_bar_sync(S.bar, S.nt);
  for (int i0 = S.tid; i0 < n; i0 += kSelBatch * S.nt) {
    uint32_t kk[kSelBatch], ix[kSelBatch];
#pragma unroll
    for (int u = 0; u < kSelBatch; ++u) {
      const int i = i0 + u * S.nt;
      kk[u] = lds_u32_if(i < n, ck_s + 4u * (uint32_t)i);
      ix[u] = lds_u32_if(i < n, ci_s + 4u * (uint32_t)i);
    }
#pragma unroll
    for (int u = 0; u < kSelBatch; ++u) {
      if (i0 + u * S.nt < n) {
        const uint32_t pos = atom_add_shared(hist_s + 4u * (kk[u] >> kHistShift), 1u);
        __stcg(gk + pos, kk[u]);
        __stcg(gi + pos, (int32_t)ix[u]);
      }
    }
  }
}

// One piece's share of a merge: (definite candidates, candidates of the cut
// bin) and the running sums of both over the pieces before it.
struct PieceCut {
  int a_pre, c_pre;
};

// Candidate f of a flat concatenation (counts given by prefix sums pre[], the
// .x or .y member) -> its piece, walking forward from *p.
template <bool kY>
__device__ __forceinline__ int piece_of(const PieceCut* pre, int nsplit, int f, int* p) {
  while (*p + 1 < nsplit && (kY ? pre[*p + 1].c_pre : pre[*p + 1].a_pre) <= f) ++*p;
  return *p;
}

// Merge the candidate blocks of one row's nsplit pieces (blocks blk0 ..
// blk0 + nsplit - 1) into its output row: the exact top-min(total, k).
// Shared memory: the row slot's buffers (ck_s, ci_s, capacity C, with the
// slot's TokSlot for the rare streaming fallback), its histogram hist_s, and
// pre (nsplit + 1 entries).  The level-1 cut comes from the pieces' summed
// histogram (`summed`, kept in L2 by a wide group's pieces) or from adding up
// the blocks' histograms.  One pass then reads every piece's prefix down to
// the cut bin: the definite candidates go to the row, the cut bin's into the
// slot with counts of their sub-bins (key bits 20..13); a split at the
// sub-bin of the row's k-th key leaves the exact selection a few candidates.
// A cut bin larger than the slot (heavy ties) is streamed through the slot.
__device__ __noinline__ void merge_pieces(const Selector S, const ScoreParams& p, int64_t blk0,
                                          int nsplit, uint32_t ck_s, uint32_t ci_s,
                                          uint32_t hist_s, TokSlot* ts, PieceCut* pre,
                                          int32_t* out_row, const uint32_t* summed = nullptr) {
  const int k = p.k;
  BinCut c{-1, 0, 0};  // bin -1: at most k candidates in all, every one definite
  if (summed) {
    // the pieces' shared histogram, searched where it lies (one pass from L2)
    c = find_bin_global(S, summed, kBins, k);
  } else {
    // summed histogram of all pieces (thread: 4-bin words tid, tid + nt, ...)
    uint32_t local = 0;
    for (int w = S.tid; w < kBins / 4; w += S.nt) {
      uint4 acc = make_uint4(0, 0, 0, 0);
      for (int sj0 = 0; sj0 < nsplit; sj0 += 8) {
        uint2 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = sj0 + u < nsplit ? __ldcg(reinterpret_cast<const uint2*>(
                                        p.cand_hist + (blk0 + sj0 + u) * kBlockBins + 4 * w))
                                  : make_uint2(0, 0);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc.x += v[u].x & 0xFFFFu; acc.y += v[u].x >> 16;
          acc.z += v[u].y & 0xFFFFu; acc.w += v[u].y >> 16;
        }
      }
      sts_v4(hist_s + 16u * (uint32_t)w, acc);
      local += acc.x + acc.y + acc.z + acc.w;
    }
    uint32_t total;
    sel_scan(S, local, &total, 1);  // also: the summed histogram is complete
    if ((int)total > k) c = find_bin(S, hist_s, kBins, k);
  }
  // per piece: definite = bins above the cut (a prefix of its block), then
  // the cut bin; every piece's two counts are loaded before they are summed
  if (S.tid < 32) {
    uint32_t ca = 0, cc = 0;
    for (int b = 0; b < nsplit; b += 128) {
      uint32_t a[4], cnt[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int sj = b + 32 * u + S.tid;
        a[u] = 0;
        cnt[u] = 0;
        if (sj < nsplit) {
          const int64_t blk = blk0 + sj;
          if (c.bin < 0) {
            a[u] = (uint32_t)__ldcg(p.cand_count + blk);
          } else {
            a[u] = __ldcg(p.cand_start + blk * kBlockBins + c.bin);
            cnt[u] = __ldcg(p.cand_hist + blk * kBlockBins + c.bin);  // 16-bit counts
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int sj = b + 32 * u + S.tid;
        const uint32_t ia = warp_inclusive_sum(a[u]), ic = warp_inclusive_sum(cnt[u]);
        if (sj < nsplit) pre[sj] = PieceCut{(int)(ca + ia - a[u]), (int)(cc + ic - cnt[u])};
        ca += __shfl_sync(0xffffffffu, ia, 31);
        cc += __shfl_sync(0xffffffffu, ic, 31);
      }
    }
    if (S.tid == 0) pre[nsplit] = PieceCut{(int)ca, (int)cc};
  }
  named_bar_sync(S.bar, S.nt);
  const int n_def = pre[nsplit].a_pre, n_cut = pre[nsplit].c_pre;
  const int need = k - n_def;
  // the cut bin's candidates: block q holds them at [definite_q, definite_q + cut_q)
  auto cut_pos = [&](int q, int f) -> int64_t {
    const int a_q = pre[q + 1].a_pre - pre[q].a_pre;
    return (blk0 + q) * p.CB + a_q + (f - pre[q].c_pre);
  };
  // One pass: the definite candidates straight to the row; the cut bin's
  // candidates, when the slot holds them, into the slot, with counts of
  // their sub-bins (key bits 20..13) in the selector's scratch.
  const bool gather = c.bin >= 0 && n_cut <= p.C;
  const uint32_t table_s = smem_u32(S.s->table);
  if (gather) {
    for (int b = S.tid; b < 256; b += S.nt) sts_u32(table_s + 4u * (uint32_t)b, 0u);
    named_bar_sync(S.bar, S.nt);
  }
  {
    // The candidates needed from piece q are a prefix of its block: its
    // a_q definite ones, then (when gathered) its c_q of the cut bin.  In
    // piece-major order piece q's run starts at e_pre(q); each lane finds the
    // piece of its element by a binary search, the searches of a batch
    // advancing together (branch-free, so their loads overlap).
    const int n_all = n_def + (gather ? n_cut : 0);
    const int lane = S.tid & 31, w = S.tid >> 5, nw = S.nt >> 5;
    int top = 1;  // the highest power of two <= nsplit
    while (2 * top <= nsplit) top *= 2;
    const uint32_t pre_s = smem_u32(pre);
    auto e_pre = [&](int q) {
      const uint2 v = lds_v2(pre_s + 8u * (uint32_t)q);
      return (int)v.x + (gather ? (int)v.y : 0);
    };
    const int units = (n_all + 31) >> 5;
    for (int j0 = w; j0 < units; j0 += nw * kMergeUnits) {
      int q[kMergeUnits], o[kMergeUnits];
      uint32_t kk[kMergeUnits];
      int32_t ix[kMergeUnits];
#pragma unroll
      for (int u = 0; u < kMergeUnits; ++u) q[u] = 0;
      for (int step = top; step > 0; step >>= 1) {
#pragma unroll
        for (int u = 0; u < kMergeUnits; ++u) {
          const int t = q[u] + step;
          const bool le = e_pre(min(t, nsplit)) <= (j0 + nw * u) * 32 + lane;  // pre[nsplit] exists
          q[u] = (le & (t < nsplit)) ? t : q[u];
        }
      }
      int a_q[kMergeUnits], d_q[kMergeUnits], c_q[kMergeUnits];  // piece's a_q, a_pre, c_pre
#pragma unroll
      for (int u = 0; u < kMergeUnits; ++u) {
        const uint2 v0 = lds_v2(pre_s + 8u * (uint32_t)q[u]);
        const uint2 v1 = lds_v2(pre_s + 8u * (uint32_t)(q[u] + 1));
        d_q[u] = (int)v0.x;
        c_q[u] = (int)v0.y;
        a_q[u] = (int)v1.x - (int)v0.x;
        o[u] = (j0 + nw * u) * 32 + lane - (d_q[u] + (gather ? c_q[u] : 0));
      }
#pragma unroll
      for (int u = 0; u < kMergeUnits; ++u) {
        const int e = (j0 + nw * u) * 32 + lane;
        kk[u] = 0u;
        ix[u] = 0;
        if (e < n_all) {
          const int64_t at = (blk0 + q[u]) * p.CB + o[u];
          ix[u] = __ldcg(p.cand_idx + at);
          if (o[u] >= a_q[u]) kk[u] = __ldcg(p.cand_keys + at);
        }
      }
#pragma unroll
      for (int u = 0; u < kMergeUnits; ++u) {
        const int e = (j0 + nw * u) * 32 + lane;
        if (e < n_all) {
          if (o[u] < a_q[u]) {
            __stcg(out_row + d_q[u] + o[u], ix[u]);
          } else {
            const uint32_t g = (uint32_t)(c_q[u] + o[u] - a_q[u]);
            sts_u32(ck_s + 4u * g, kk[u]);
            sts_u32(ci_s + 4u * g, (uint32_t)ix[u]);
            red_add_shared_if(true, table_s + 4u * ((kk[u] >> 13) & 255u), 1u);
          }
        }
      }
    }
  }
  if (c.bin < 0) {
    for (int i = n_def + S.tid; i < k; i += S.nt) __stcg(out_row + i, -1);
    return;
  }
  if (gather) {
    named_bar_sync(S.bar, S.nt);  // the gathered candidates and their sub-bin counts
    // the sub-bin of the need-th largest: the higher sub-bins go to the row,
    // that sub-bin is selected exactly
    const BinCut c2 = find_bin_warp(table_s, 256, need);
    const uint32_t lo = ((uint32_t)c.bin << kHistShift) | ((uint32_t)c2.bin << 13);
    const int2 r = split_pass(S, n_cut, ck_s, ci_s, lo, (uint64_t)lo + (1ull << 13), out_row + n_def,
                              need);
    const int above = min(r.x, need), rest = need - above;
    if (rest <= 0) return;
    if (r.y <= S.nt) {
      rank_small(S, r.y, ck_s, ci_s, rest, out_row + n_def + above);
    } else {
      const BinCut cut{c.bin, 0, r.y};
      slot_select(S, kSelRow, r.y, ck_s, ci_s, hist_s, rest, 0, nullptr, out_row + n_def + above,
                  nullptr, &cut);
    }
    return;
  }
  // Rare: more cut-bin candidates than the slot holds (heavily tied scores).
  // Stream them through the slot, shrinking it to the top `need` as it fills.
  clear_bins(S, hist_s, kBins);
  if (S.tid == 0) {
    ts->count = 0;
    ts->thr = 0u;
  }
  named_bar_sync(S.bar, S.nt);
  uint32_t* ck = reinterpret_cast<uint32_t*>(__cvta_shared_to_generic(ck_s));
  int32_t* ci = reinterpret_cast<int32_t*>(__cvta_shared_to_generic(ci_s));
  const int batch = S.nt;
  int sj = 0;
  for (int f0 = 0; f0 < n_cut; f0 += batch) {
    const int f = f0 + S.tid;
    const uint32_t thr = ts->thr;
    uint32_t key = 0u;
    int32_t idx = 0;
    if (f < n_cut) {
      const int64_t o = cut_pos(piece_of<true>(pre, nsplit, f, &sj), f);
      key = __ldcg(p.cand_keys + o);
      idx = __ldcg(p.cand_idx + o);
    }
    slot_append(key, idx, thr, ts, ck, ci, hist_s);
    named_bar_sync(S.bar, S.nt);
    const int n = ts->count;
    if (n > p.C - batch) {
      uint32_t nthr = 0;
      const int kept =
          slot_select(S, kSelInPlace, n, ck_s, ci_s, hist_s, need, p.C - batch, nullptr, nullptr, &nthr);
      if (S.tid == 0) {
        ts->count = kept;
        ts->thr = nthr;
      }
      named_bar_sync(S.bar, S.nt);
    }
  }
  slot_select(S, kSelRow, ts->count, ck_s, ci_s, hist_s, need, 0, nullptr, out_row + n_def, nullptr);
}

// An Item loaded where the call stands (see ld_ahead).
__device__ __forceinline__ Item item_of(int4 a, int4 b) {
  Item I;
  I.r = a.x;
  I.t0 = a.y;
  I.gcount = a.z;
  I.k0 = a.w;
  I.k1 = b.x;
  I.split = b.y;
  I.cand_block = b.z;
  I.sgroup = b.w;
  return I;
}
__device__ __forceinline__ Item load_item(const Item* items, int i) {
  return item_of(ld_ahead_v4(items + i), ld_ahead_v4(reinterpret_cast<const int4*>(items + i) + 1));
}

// sum_h wq[h] * ReLU(acc[h]) over the H accumulator columns at taddr (this
// thread's TMEM lane); wq_s is the shared-memory address of the H weights.
// The weights are read (explicit shared loads) before the tensor-memory
// wait; the products are accumulated pairwise with the packed two-lane FMA
// (fma.rn.f32x2: two FP32 FMAs per instruction, each rounded as fmaf), in
// four pair accumulators so that the FMA chains stay short.
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack_f32x2(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

template <int H>
__device__ __forceinline__ float relu_weighted_sum(uint32_t taddr, uint32_t wq_s) {
  constexpr int CH = H >= 32 ? 32 : H;              // columns per tcgen05.ld
  constexpr int BATCH = H >= 64 ? 64 : H;           // columns loaded before one wait
  constexpr int NA = BATCH >= 16 ? 4 : BATCH / 4;   // pair accumulators
  unsigned long long acc[NA];
#pragma unroll
  for (int i = 0; i < NA; ++i) acc[i] = 0ull;
#pragma unroll
  for (int c0 = 0; c0 < H; c0 += BATCH) {
    uint4 ww[BATCH / 4];
#pragma unroll
    for (int i = 0; i < BATCH / 4; ++i) ww[i] = lds_v4(wq_s + 4u * (uint32_t)(c0 + 4 * i));
    uint32_t v[BATCH];
#pragma unroll
    for (int c = 0; c < BATCH; c += CH) tmem_ld<CH>(taddr + c0 + c, v + c);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < BATCH; h += 4) {
      unsigned long long& a = acc[(h / 4) % NA];
      a = fma_f32x2(pack_f32x2(__uint_as_float(ww[h / 4].x), __uint_as_float(ww[h / 4].y)),
                    pack_f32x2(fmaxf(__uint_as_float(v[h + 0]), 0.f),
                               fmaxf(__uint_as_float(v[h + 1]), 0.f)),
                    a);
      a = fma_f32x2(pack_f32x2(__uint_as_float(ww[h / 4].z), __uint_as_float(ww[h / 4].w)),
                    pack_f32x2(fmaxf(__uint_as_float(v[h + 2]), 0.f),
                               fmaxf(__uint_as_float(v[h + 3]), 0.f)),
                    a);
    }
  }
  float2 t = unpack_f32x2(acc[0]);
  float sum = t.x + t.y;
#pragma unroll
  for (int i = 1; i < NA; ++i) {
    t = unpack_f32x2(acc[i]);
    sum += t.x + t.y;
  }
  return sum;
}

// The same sums for two blocks at once (TMEM column bases ta and tb, same
// weights): the two FMA chains are independent, so each hides the other's
// latency, and the weights are read once for both.  Columns go in chunks of
// 32 per block so that both chunks and their weights stay in registers.
template <int H>
__device__ __forceinline__ float2 relu_weighted_sum2(uint32_t ta, uint32_t tb, uint32_t wq_s) {
  constexpr int CH = H >= 32 ? 32 : H;             // columns per chunk and block
  constexpr int NA = CH >= 16 ? 4 : CH / 4;        // pair accumulators per block
  unsigned long long aa[NA], ab[NA];
#pragma unroll
  for (int i = 0; i < NA; ++i) aa[i] = ab[i] = 0ull;
#pragma unroll
  for (int c0 = 0; c0 < H; c0 += CH) {
    uint4 ww[CH / 4];
#pragma unroll
    for (int i = 0; i < CH / 4; ++i) ww[i] = lds_v4(wq_s + 4u * (uint32_t)(c0 + 4 * i));
    uint32_t va[CH], vb[CH];
    tmem_ld<CH>(ta + c0, va);
    tmem_ld<CH>(tb + c0, vb);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < CH; h += 4) {
      const unsigned long long w01 =
          pack_f32x2(__uint_as_float(ww[h / 4].x), __uint_as_float(ww[h / 4].y));
      const unsigned long long w23 =
          pack_f32x2(__uint_as_float(ww[h / 4].z), __uint_as_float(ww[h / 4].w));
      unsigned long long& a = aa[(h / 4) % NA];
      unsigned long long& b = ab[(h / 4) % NA];
      a = fma_f32x2(w01, pack_f32x2(fmaxf(__uint_as_float(va[h]), 0.f),
                                    fmaxf(__uint_as_float(va[h + 1]), 0.f)), a);
      b = fma_f32x2(w01, pack_f32x2(fmaxf(__uint_as_float(vb[h]), 0.f),
                                    fmaxf(__uint_as_float(vb[h + 1]), 0.f)), b);
      a = fma_f32x2(w23, pack_f32x2(fmaxf(__uint_as_float(va[h + 2]), 0.f),
                                    fmaxf(__uint_as_float(va[h + 3]), 0.f)), a);
      b = fma_f32x2(w23, pack_f32x2(fmaxf(__uint_as_float(vb[h + 2]), 0.f),
                                    fmaxf(__uint_as_float(vb[h + 3]), 0.f)), b);
    }
  }
  float2 r = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < NA; ++i) {
    const float2 ta2 = unpack_f32x2(aa[i]), tb2 = unpack_f32x2(ab[i]);
    r.x += ta2.x + ta2.y;
    r.y += tb2.x + tb2.y;
  }
  return r;
}

template <int H>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_topk_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_s,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ ScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  // align to 1024 by pointer arithmetic on the shared array itself, so the
  // compiler keeps every access below in the shared address space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint8_t* stage_base = smem + p.off_stage;
  const uint32_t scale_ring_s = smem_u32(smem + p.off_scale);
  uint8_t* q_base = smem + p.off_q;
  uint32_t* ckeys_all = reinterpret_cast<uint32_t*>(smem + p.off_ckeys);
  int32_t* cidx_all = reinterpret_cast<int32_t*>(smem + p.off_cidx);
  float* wq_all = reinterpret_cast<float*>(smem + p.off_wq);
  TokSlot* tok = reinterpret_cast<TokSlot*>(smem + p.off_tok);
  int* hist_all = reinterpret_cast<int*>(smem + p.off_hist);
  Misc* misc = reinterpret_cast<Misc*>(smem + p.off_misc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  const uint32_t bar_full = smem_u32(bars);
  const uint32_t bar_empty = bar_full + 8 * kMaxStages;
  const uint32_t bar_tfull = bar_empty + 8 * kMaxStages;
  const uint32_t bar_tempty = bar_tfull + 8 * kMaxAccBufs;
  const uint32_t bar_qfull = bar_tempty + 8 * kMaxAccBufs;
  const uint32_t bar_qempty = bar_qfull + 8 * kMaxQBufs;
  const uint32_t bar_drain = bar_qempty + 8 * kMaxQBufs;
  volatile int* abort_flag = &misc->abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      // one arrival (with its expected bytes) per page of the tile
      mbar_init(bar_full + 8 * s, 2 * p.BPS);
      mbar_init(bar_empty + 8 * s, 1);  // freed by the MMA commit
    }
    for (int b = 0; b < p.NB; ++b) {
      // the MMA commit plus the issuing thread's own arrival (which publishes the
      // tile's scales, observed through the full barrier, to the epilogue)
      mbar_init(bar_tfull + 8 * b, 2);
      // decode layout with one block per tile: one warpgroup reads a tile;
      // otherwise both do (each warp arrives once per tile)
      mbar_init(bar_tempty + 8 * b, (p.G == 1 && p.BPS == 1) ? kEpiWarps / 2 : kEpiWarps);
    }
    for (int b = 0; b < p.NQ; ++b) {
      mbar_init(bar_qfull + 8 * b, 1);
      mbar_init(bar_qempty + 8 * b, 1);
    }
    mbar_init(bar_drain, 1);
    misc->abort = 0;
    misc->epi_abort = 0;
    misc->merge_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_s);
    tma_prefetch_desc(&tm_q);
  }
  // Keys per tile and the producer's view of a chunk of an item's page ids:
  // lane l holds page 32 * chunk + l of the item, -1 where the item has none.
  const int KS = kTileKeys * p.BPS;
  const int ppt = 2 * p.BPS;  // pages per tile
  const int tpc = 32 / ppt;   // tiles per 32-page chunk
  auto tiles_of = [&](const Item& J) { return (J.k1 - J.k0 + KS - 1) / KS; };
  auto in_range = [&](const Item& J, int chunk) {
    return chunk * tpc < tiles_of(J) && (J.k0 / kPageTokens + chunk * 32 + lane) * kPageTokens < J.k1;
  };
  auto fetch = [&](const Item& J, int chunk) -> int32_t {
    return in_range(J, chunk)
               ? ld_ahead(p.block_table + (int64_t)J.r * p.max_blocks + J.k0 / kPageTokens + chunk * 32 + lane)
               : -1;
  };
  // Entries below stable_end of an item's request are not written by the
  // preceding cache write: its new tokens sit at positions >= seq_len - q_len,
  // and an entry e is written only by a position >= e * ratio.
  const bool early = p.meta_ready != 0;
  auto stable_end_of = [&](const Item& J) -> int {
    if (!early) return 0;
    const int q_len = ld_ahead(p.qsl + J.r + 1) - ld_ahead(p.qsl + J.r);
    return (ld_ahead(p.seq_lens + J.r) - q_len) / p.ratio;
  };
  // The producer's first three items with the page ids of their first chunks
  // and their stable ends.  Inputs (block table, query_start_loc, seq_lens)
  // and, with meta_ready, the plan's outputs are complete before this kernel
  // starts, so these loads overlap the preceding kernel.  (Once the page copies
  // of every SM are in flight, any load takes microseconds, so nothing the
  // producer needs for a decode CTA's items is loaded later.)
  int it_begin = 0, it_end = 0;
  Item I_cur{}, I_next{}, I_after{};
  int32_t raw_cur = -1, raw_next = -1, raw_after = -1;
  int se_cur = 0, se_next = 0, se_after = 0;
  auto load_meta = [&] {
    const int4* head = reinterpret_cast<const int4*>(p.heads + blockIdx.x);
    const int4 range = ld_ahead_v4(head + 2);
    it_begin = range.x;
    it_end = range.y;
    if (warp == 0) {
      if (it_begin < it_end) I_cur = item_of(ld_ahead_v4(head), ld_ahead_v4(head + 1));
      if (it_begin + 1 < it_end) I_next = load_item(p.items, it_begin + 1);
      if (it_begin + 2 < it_end) I_after = load_item(p.items, it_begin + 2);
      if (it_begin < it_end) {
        raw_cur = fetch(I_cur, 0);
        se_cur = stable_end_of(I_cur);
      }
      if (it_begin + 1 < it_end) {
        raw_next = fetch(I_next, 0);
        se_next = stable_end_of(I_next);
      }
      if (it_begin + 2 < it_end) {
        raw_after = fetch(I_after, 0);
        se_after = stable_end_of(I_after);
      }
    }
  };
  if (early) load_meta();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // everything above overlaps the preceding kernel (plan or cache write) when
  // launched with programmatic stream serialisation; its outputs are read
  // below.  With meta_ready the producer waits later, only before what the
  // preceding kernel may write.
  if (!(early && warp == 0)) pdl_wait();
  // every block of this persistent grid is resident: the row kernel's blocks
  // may be placed as SMs free up (they wait for this grid's completion)
  pdl_launch_dependents();
  if (!early) load_meta();
  const uint32_t tmem_base = misc->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the tiles.  Per tile, lane 0 waits for the stage
    // (from the NS-th tile on; the first NS stages start free); then each lane
    // that holds one of the tile's page ids arrives on the stage's full
    // barrier with that page's bytes and issues two copies: the page's 64 key
    // rows (8 KB, 128-byte swizzle, into the stage) and its 256 bytes of
    // scales (into the tile's slot of the scale ring).  A lane whose page is
    // missing (beyond the item, or outside the pool) writes zero scales (a
    // zero scale marks its keys invalid) and arrives without bytes.  Tile s
    // uses scale slot s % NR with NR >= NS + NB: the producer reaches tile s
    // only after the epilogue has released tile s - NS - NB, so a slot is
    // never overwritten while read.  NB and NR are powers of two, so the
    // per-tile ring positions are masks and shifts (a 64-bit division by a
    // runtime value costs hundreds of cycles of dependent instructions on the
    // per-tile path).
    // The page ids of the next 32 pages come from one coalesced load (lane l
    // holds page 32 * chunk + l of the item), fetched one chunk ahead.
    // Items are pipelined three deep: the current item and the next two are
    // held with their first chunk's page ids; the item three ahead is loaded
    // once the current item's first tile is issued, and its page ids when the
    // current item ends.
    // With meta_ready the warp streams the tiles whose pages are stable before
    // the programmatic-launch wait, and waits before the first tile that may
    // hold a new entry or may have to wait for a free stage (seq >= NS), and,
    // unless q_ready, before the first query load (deferred until then).
    int stage = 0;
    uint32_t sphase = 0;
    int q_last[kMaxQBufs] = {-1, -1};
    int item_i = 0;
    long long seq = 0;  // tile sequence number of this CTA (all roles count alike)
    bool ok = true;
    bool waited = !early;
    auto ensure_wait = [&] {
      if (!waited) {
        pdl_wait();
        waited = true;
      }
    };
    const uint32_t stage_bytes = (uint32_t)(p.BPS * kStageBytes);
    const uint32_t slot_bytes = (uint32_t)(p.BPS * kScaleSlotBytes);
    constexpr int kPageScaleBytes = kPageTokens * 4;  // 256: rows 64 and 65 of the page
    Item I_far{};
    // a decode batch (one query row per group) reads every page once per
    // launch: its lines go first from L2, so that the launch's metadata,
    // candidate blocks and code stay
    const bool read_once = p.G == 1;
    const uint64_t l2_once = l2_policy_evict_first();
    for (int it = it_begin; it < it_end && ok; ++it, ++item_i) {
      const Item I = I_cur;
      const int stable_end = se_cur;
      const int qb = item_i % p.NQ;
      const uint32_t qpar = (uint32_t)((item_i / p.NQ) & 1);
      int okv = 1;
      // the first NQ query buffers are free from the start
      if (lane == 0 && item_i >= p.NQ) okv = mbar_wait(bar_qempty + 8 * qb, qpar ^ 1, abort_flag, p.wait_limit);
      if (!__shfl_sync(0xffffffffu, okv, 0)) { ok = false; break; }
      bool q_pending = true;
      auto issue_q = [&] {
        q_pending = false;
        q_last[qb] = item_i;
        if (lane == 0) {
          uint8_t* q_tile = q_base + qb * p.q_bytes;
          if (p.q_box_per_token) {
            mbar_arrive_expect_tx(bar_qfull + 8 * qb, (uint32_t)(I.gcount * H * kHeadDim));
            for (int g = 0; g < I.gcount; ++g)
              tma_load_2d(smem_u32(q_tile + g * H * kHeadDim), &tm_q, 0, (I.t0 + g) * H,
                          bar_qfull + 8 * qb);
          } else {
            mbar_arrive_expect_tx(bar_qfull + 8 * qb, (uint32_t)(p.G * H * kHeadDim));
            tma_load_2d(smem_u32(q_tile), &tm_q, 0, I.t0 * H, bar_qfull + 8 * qb);
          }
        }
      };
      // item 0's first tile is issued before its queries (the tile's pages
      // take longer to arrive than the queries)
      if (item_i > 0 && (p.q_ready || waited)) issue_q();
      const int ntiles = tiles_of(I);
      int32_t raw = raw_cur;
      bool ahead = false;  // the next items' loads were issued
      for (int c = 0; c * tpc < ntiles && ok; ++c) {
        int32_t cur = -1;  // this lane's page of the chunk, -1 if none or invalid
        if (in_range(I, c)) {
          if (raw >= 0 && (int64_t)raw < p.num_pages) cur = raw;
          else raise_status(p.status, kStatusBadPage);
        }
        raw = fetch(I, c + 1);
        const int jend = min(tpc, ntiles - c * tpc);
        for (int jj = 0; jj < jend; ++jj, ++seq) {
          // the tile's pages are held by chunk lanes first .. first + ppt - 1,
          // and those lanes issue their own page copies
          const int first = ppt * jj;
          const bool mine = lane >= first && lane < first + ppt;
          if (!waited) {
            // the tile's pages end at a page boundary: all of them below stable_end?
            const int tile_end = min(I.k0 + (c * tpc + jj + 1) * KS, I.k1);
            const int page_end = (tile_end + kPageTokens - 1) / kPageTokens * kPageTokens;
            if (seq >= p.NS || page_end > stable_end) ensure_wait();
          }
          if (q_pending && (p.q_ready || waited) && (item_i > 0 || seq > 0)) issue_q();
          okv = 1;
          // the first NS stages are free from the start
          if (lane == 0 && seq >= p.NS) okv = mbar_wait(bar_empty + 8 * stage, sphase ^ 1, abort_flag, p.wait_limit);
          if (!__shfl_sync(0xffffffffu, okv, 0)) { ok = false; break; }
          if (mine) {
            const uint32_t pi = (uint32_t)(lane - first);  // page of the tile
            const uint32_t sdst = scale_ring_s + ((uint32_t)seq & (uint32_t)(p.NR - 1)) * slot_bytes +
                                  pi * (uint32_t)kPageScaleBytes;
            const uint32_t full = bar_full + 8 * stage;
            if (cur >= 0) {
              mbar_arrive_expect_tx(full, (uint32_t)(kPageTokens * kHeadDim + kPageScaleBytes));
              const int32_t row = cur * (kPageBytes / kHeadDim);  // the page's first 128-byte row
              const uint32_t kdst = smem_u32(stage_base) + (uint32_t)stage * stage_bytes +
                                    pi * (uint32_t)(kPageTokens * kHeadDim);
              if (read_once) {
                tma_load_2d_hint(kdst, &tm_k, 0, row, full, l2_once);
                tma_load_2d_hint(sdst, &tm_s, 0, row + kPageTokens, full, l2_once);
              } else {
                tma_load_2d(kdst, &tm_k, 0, row, full);
                tma_load_2d(sdst, &tm_s, 0, row + kPageTokens, full);
              }
            } else {
              for (uint32_t i = 0; i < (uint32_t)kPageScaleBytes; i += 16u) sts_v4(sdst + i, make_uint4(0u, 0u, 0u, 0u));
              mbar_arrive(full);
            }
          }
          __syncwarp();
          if (++stage == p.NS) { stage = 0; sphase ^= 1; }
          if (!ahead) {
            ahead = true;
            if (it + 3 < it_end) I_far = load_item(p.items, it + 3);
          }
        }
      }
      if (!ahead && it + 3 < it_end) I_far = load_item(p.items, it + 3);  // an item without tiles
      if (q_pending && ok) {  // an item whose tiles all went out before its queries
        if (!p.q_ready) ensure_wait();
        issue_q();
      }
      I_cur = I_next;
      raw_cur = raw_next;
      se_cur = se_next;
      I_next = I_after;
      raw_next = raw_after;
      se_next = se_after;
      I_after = I_far;
      if (it + 3 < it_end) {
        raw_after = fetch(I_far, 0);
        se_after = stable_end_of(I_far);
      }
    }
    ensure_wait();
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, kStatusTimeout);
      }
      // never leave with bulk copies in flight into this CTA's shared memory:
      // wait for the last tile issued on every stage (tiles 0 .. seq-1, tile t
      // on stage t % NS in phase (t / NS) & 1)
      for (int s = 0; s < p.NS; ++s) {
        if (seq > s) {
          const long long t_last = s + (long long)p.NS * ((seq - 1 - s) / p.NS);
          mbar_wait(bar_full + 8 * s, (uint32_t)((t_last / p.NS) & 1), nullptr);
        }
      }
      for (int b = 0; b < p.NQ; ++b)
        if (q_last[b] >= 0) mbar_wait(bar_qfull + 8 * b, (uint32_t)((q_last[b] / p.NQ) & 1), nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t sphase = 0, aphase = 0;
      int item_i = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it, ++item_i) {
        const Item I = p.items[it];
        const uint32_t N = (uint32_t)((I.gcount * H + 15) & ~15);
        const uint32_t idesc = idesc_e4m3_f32(128, N);
        const int qb = item_i % p.NQ;
        if (!mbar_wait(bar_qfull + 8 * qb, (uint32_t)((item_i / p.NQ) & 1), abort_flag,
                       p.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t qaddr = smem_u32(q_base + qb * p.q_bytes);
        const int ntiles = (I.k1 - I.k0 + kTileKeys * p.BPS - 1) / (kTileKeys * p.BPS);
        for (int j = 0; j < ntiles; ++j) {
          if (!mbar_wait(bar_full + 8 * stage, sphase, abort_flag, p.wait_limit)) { ok = false; break; }
          if (!mbar_wait(bar_tempty + 8 * acc, aphase ^ 1, abort_flag, p.wait_limit)) { ok = false; break; }
          tc_fence_after();
          mbar_arrive(bar_tfull + 8 * acc);  // the tile's scales (seen via full) are ready
          const uint32_t aaddr = smem_u32(stage_base) + (uint32_t)(stage * p.BPS * kStageBytes);
          const uint32_t d = tmem_base + (uint32_t)(acc * p.BPS * p.n_max);
          for (int b = 0; b < p.BPS; ++b) {
#pragma unroll
            for (int kk = 0; kk < kHeadDim / 32; ++kk)
              umma_f8(d + (uint32_t)(b * p.n_max),
                      sw128_desc(aaddr + (uint32_t)(b * kStageBytes) + kk * 32),
                      sw128_desc(qaddr + kk * 32), idesc, kk > 0);
          }
          umma_commit(bar_empty + 8 * stage);
          umma_commit(bar_tfull + 8 * acc);
          if (++stage == p.NS) { stage = 0; sphase ^= 1; }
          if (++acc == p.NB) { acc = 0; aphase ^= 1; }
        }
        if (!ok) break;
        umma_commit(bar_qempty + 8 * qb);
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, kStatusTimeout);
      }
      // wait for every MMA this thread issued before tensor memory is released
      umma_commit(bar_drain);
      mbar_wait(bar_drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Thread = one key row of a tile (its TMEM lane).  With one query row per
    // item (decode) the two warpgroups take alternate tiles and share the
    // row's candidate buffer; otherwise each warpgroup owns alternate rows of
    // the group and both read every tile.  Each thread reads its key's scale
    // from the tile's slot of the scale ring.
    const int epi = warp - 2;          // 0..7
    const int wg = epi >> 2;           // warpgroup 0/1
    const int tid = (epi & 3) * 32 + lane;
    const int quad = warp & 3;         // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;  // key row of the tile = TMEM lane
    const bool alt = (p.G == 1);
    const int step = alt ? 2 : 1;
    // who selects a row's candidates: both warpgroups for a decode row, else its warpgroup
    const Selector S = alt ? Selector{256, epi * 32 + lane, 3u, nullptr, &misc->sel[0]}
                           : Selector{128, tid, 1u + wg, nullptr, &misc->sel[wg]};
    // level-1 histogram of each row slot's candidates (2048 bins per slot)
    const uint32_t hist0_s = smem_u32(hist_all);
    auto hist_of = [&](int g) -> uint32_t { return hist0_s + (uint32_t)g * kBins * 4u; };
    auto ck_of = [&](int g) -> uint32_t* { return ckeys_all + (size_t)g * p.C; };
    auto ci_of = [&](int g) -> int32_t* { return cidx_all + (size_t)g * p.C; };
    auto out_row = [&](int g) -> int32_t* { return p.topk + (int64_t)tok[g].t * p.k; };
    // Buffer-fill checks: the rows' warps append at most kpi keys per
    // iteration, so the next check comes after as many iterations as the
    // fullest row's free room holds (at most 32); a row with less free room
    // than `headroom` shrinks to a superset of its top-k first (keeping at
    // most C - headroom), so checks stay at least headroom / kpi apart.
    const int kpi = kTileKeys * (alt ? 2 : 1);
    const int headroom = (p.C - 8 * kpi >= 2 * p.k ? 8 : 4) * kpi;
    long long tile_base = 0;  // tiles of earlier items of this CTA (all roles count alike)
    bool ok = true;
    const int g_first = alt ? 0 : wg;  // this thread's rows: g_first, g_first + 2, ...
    const bool sets_up = !alt || wg == 0;  // per-row setup: warpgroup 0 for the shared decode row
    for (int it = it_begin; it < it_end && ok; ++it) {
      const Item I = p.items[it];
      const int qb0 = __ldg(p.qsl + I.r);
      const int q_len = __ldg(p.qsl + I.r + 1) - qb0;
      const int seq_len = __ldg(p.seq_lens + I.r);
      const int nsplit = I.split >> 16;
      const int split = I.split & 0xFFFF;
      const bool to_rows = I.sgroup == kSgroupRows;  // keys to the workspace, selected later
      // A row cut into many pieces shares a histogram of its candidates' level-1
      // bins: each piece adds its own once, at its first fill check, and at its
      // first three checks raises its admission threshold to the bin where that
      // histogram's count from the top reaches k.  The histogram counts distinct
      // keys of the row (each piece publishes once, pieces are disjoint), so at
      // least k keys of the row lie in or above that bin: no key below it is
      // among the row's top k, in any piece.  Pieces that publish late only make
      // the bound weaker.  The pieces also sum their final candidates' bins
      // into a second shared histogram, which the merge reads instead of
      // adding up every piece's.
      const int wid = (!to_rows && nsplit >= kWideSplit && p.G == 1) ? __ldg(p.wide_of + I.sgroup) : -1;
      const bool wide = wid >= 0;
      int gstate = 0;  // checks done since the item began (wide items publish at the first)
      auto early_hist = [&](int) { return p.ghist + (int64_t)wid * kSharedHistWords; };
      auto final_hist = [&](int g) { return early_hist(g) + kBins; };
      for (int g = g_first; g < I.gcount; g += 2) {
        const int t = I.t0 + g;
        if (sets_up) {
          for (int h = tid; h < H; h += 128)
            wq_all[g * H + h] =
                __ldg(p.w + (int64_t)t * H + h) * __ldg(p.q_scale + (int64_t)t * H + h);
          if (tid == 0) {
            tok[g].count = 0;
            tok[g].thr = 0u;
            tok[g].pos = (seq_len - q_len + (t - qb0) + 1) / p.ratio - 1;  // last visible entry
            tok[g].t = t;
          }
        }
      }
      for (int g = g_first; g < I.gcount; g += 2) clear_bins(S, hist_of(g), kBins);
      named_bar_sync(3, 256);
      const int ntiles = (I.k1 - I.k0 + KS - 1) / KS;
      const int units = ntiles * p.BPS;  // 128-key blocks of the item
      const bool may_fill = !to_rows && (I.k1 - I.k0) > p.C;
      const int u0 = alt ? wg : 0;
      const int iters = alt ? (units + 1) / 2 : units;
      // This warpgroup's blocks go two at a time (iterations m and m + 1):
      // their head sums interleave (two independent FMA chains per thread)
      // and share the weight loads, and each pair pays the loop's waits and
      // fences once.  Fill checks come after pairs: `next_chk` is the pair
      // after which the next one runs; a wide item checks after its 2nd and
      // 4th pair, so that its pieces share their bound early.
      int next_chk = wide ? 1 : max(0, min(16, p.C / (2 * kpi)) - 1);
      for (int m = 0; m < iters; m += 2) {
        const int uA = u0 + m * step, uB = uA + step;  // block u = (tile j, block b of the tile)
        const bool hasA = uA < units;
        const bool hasB = hasA && m + 1 < iters && uB < units;
        const int jA = uA >> p.lg_bps, bA = uA & (p.BPS - 1);
        const int jB = uB >> p.lg_bps, bB = uB & (p.BPS - 1);
        const long long seqA = tile_base + jA, seqB = tile_base + jB;
        const int accA = (int)((uint32_t)seqA & (uint32_t)(p.NB - 1));
        const int accB = (int)((uint32_t)seqB & (uint32_t)(p.NB - 1));
        if (hasA && ok) {
          const int keyA = I.k0 + jA * KS + bA * kTileKeys + row;
          const int keyB = I.k0 + jB * KS + bB * kTileKeys + row;
          // no early exit on the abort flag here: the warps of a warpgroup must take
          // the same branch, so they all wait on the same phase with the same limit
          if (!mbar_wait(bar_tfull + 8 * accA, (uint32_t)(seqA >> p.lg_nb) & 1u, nullptr,
                         p.wait_limit))
            ok = false;
          if (ok && hasB &&
              !mbar_wait(bar_tfull + 8 * accB, (uint32_t)(seqB >> p.lg_nb) & 1u, nullptr,
                         p.wait_limit))
            ok = false;
          if (ok) {
            tc_fence_after();
            // the keys' scales; zero (never a written scale) for a page outside the pool
            const uint32_t slot_b = (uint32_t)(p.BPS * kScaleSlotBytes);
            const float scA = __uint_as_float(
                lds_u32(scale_ring_s + ((uint32_t)seqA & (uint32_t)(p.NR - 1)) * slot_b +
                        (uint32_t)(bA * kTileKeys + row) * 4u));
            const float scB = hasB ? __uint_as_float(lds_u32(
                                         scale_ring_s + ((uint32_t)seqB & (uint32_t)(p.NR - 1)) * slot_b +
                                         (uint32_t)(bB * kTileKeys + row) * 4u))
                                   : 0.f;
            const bool kvalidA = scA > 0.f && keyA < I.k1;
            const bool kvalidB = hasB && scB > 0.f && keyB < I.k1;
            const uint32_t lanes = tmem_base + ((uint32_t)(quad * 32) << 16);
            const uint32_t tA = lanes + (uint32_t)((accA * p.BPS + bA) * p.n_max);
            // without a second block the pair's second sum repeats the first (unused)
            const uint32_t tB = hasB ? lanes + (uint32_t)((accB * p.BPS + bB) * p.n_max) : tA;
            // the pair's accumulators go back to the MMA as soon as this warp's
            // last tensor-memory read of them is done (before its appends)
            bool released = false;
            auto release = [&] {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                mbar_arrive(bar_tempty + 8 * accA);
                if (hasB) mbar_arrive(bar_tempty + 8 * accB);
              }
              released = true;
            };
            for (int g = g_first; g < I.gcount; g += 2) {
              const float2 sum = relu_weighted_sum2<H>(tA + (uint32_t)(g * H), tB + (uint32_t)(g * H),
                                                       smem_u32(wq_all + g * H));
              if (g + 2 >= I.gcount) release();
              const float scoreA = sum.x * scA, scoreB = sum.y * scB;
              const int pos = tok[g].pos;
              const bool validA = kvalidA && keyA <= pos, validB = kvalidB && keyB <= pos;
              if (p.scores_out) {
                if (validA && keyA < p.scores_ld) p.scores_out[(int64_t)tok[g].t * p.scores_ld + keyA] = scoreA;
                if (validB && keyB < p.scores_ld) p.scores_out[(int64_t)tok[g].t * p.scores_ld + keyB] = scoreB;
              }
              const uint32_t kkA = validA ? score_key(scoreA) : 0u;
              const uint32_t kkB = validB ? score_key(scoreB) : 0u;
              if (to_rows) {
                uint32_t* srow = p.score_rows + (int64_t)tok[g].t * p.score_stride;
                if (keyA < I.k1) srow[keyA] = kkA;
                if (hasB && keyB < I.k1) srow[keyB] = kkB;
              } else {
                slot_append2(kkA, keyA, kkB, keyB, tok[g].thr, &tok[g],
                             ckeys_all + (size_t)g * p.C, cidx_all + (size_t)g * p.C, hist_of(g));
              }
            }
            if (!released) release();  // a warpgroup without a row in this item
          }
        }
        const bool check = may_fill && m / 2 == next_chk && m + 2 < iters;
        if (check) {
          // the row's appending warps only (its warpgroup, or both for a decode row)
          if (!ok) misc->epi_abort = 1;
          named_bar_sync(S.bar, S.nt);  // every append so far is visible
          if (misc->epi_abort) {
            ok = false;
          } else {
            for (int g = g_first; g < I.gcount; g += 2) {
              const int n = tok[g].count;
              if (n > p.C - headroom) {
                uint32_t thr = 0;
                const int kept = slot_select(S, kSelInPlace, n, smem_u32(ck_of(g)),
                                             smem_u32(ci_of(g)), hist_of(g), p.k, p.C - headroom,
                                             nullptr, nullptr, &thr);
                if (S.tid == 0) {
                  tok[g].count = kept;
                  tok[g].thr = thr;
                }
              }
            }
            if (wide && gstate == 0) {
              named_bar_sync(S.bar, S.nt);  // the histograms are current
              for (int g = g_first; g < I.gcount; g += 2) {
                uint32_t* gh = early_hist(g);
                for (int b = S.tid; b < kBins; b += S.nt) {
                  const uint32_t c = lds_u32(hist_of(g) + 4u * (uint32_t)b);
                  if (c) atomicAdd(gh + b, c);
                }
              }
            }
            if (wide && gstate < 3) {
              // adopt the shared bound (at the first three checks: it only rises
              // as the other pieces publish) as the admission threshold; the
              // candidates already held below it stay until the next shrink
              // (they are keys of the row, so any superset kept stays valid)
              for (int g = g_first; g < I.gcount; g += 2) {
                const BinCut c = find_bin_global(S, early_hist(g), kBins, p.k);
                const uint32_t gthr = c.bin > 0 ? ((uint32_t)c.bin << kHistShift) - 1u : 0u;
                if (S.tid == 0 && gthr > tok[g].thr) tok[g].thr = gthr;
              }
            }
            ++gstate;
          }
          named_bar_sync(S.bar, S.nt);
          int room = p.C;
          for (int g = g_first; g < I.gcount; g += 2) room = min(room, p.C - tok[g].count);
          // the pairs until the next check: as many as the free room holds
          next_chk = m / 2 + max(1, min(wide && gstate < 2 ? 2 : 16, room / (2 * kpi)));
        }
      }
      tile_base += ntiles;
      if (!ok) misc->epi_abort = 1;
      named_bar_sync(3, 256);  // every append of the item is done
      if (misc->epi_abort) { ok = false; break; }
      // finalize this item's rows (rows scored into the workspace are
      // selected by the row kernel)
      for (int g = g_first; g < I.gcount && !to_rows; g += 2) {
        const int n0 = tok[g].count;
        if (nsplit == 1) {
          select_row(S, n0, smem_u32(ck_of(g)), smem_u32(ci_of(g)), hist_of(g), p.k, out_row(g));
        } else {
          // a superset of the piece's top-k, at most one block
          const int64_t blk = (int64_t)I.cand_block + (int64_t)g * nsplit + split;
          int n = n0;
          if (n > p.CB) {
            uint32_t thr = 0;
            n = slot_select(S, kSelInPlace, n, smem_u32(ck_of(g)), smem_u32(ci_of(g)), hist_of(g),
                            p.k, p.CB, nullptr, nullptr, &thr);
          }
          slot_emit_sorted(S, n, smem_u32(ck_of(g)), smem_u32(ci_of(g)), hist_of(g),
                           p.cand_keys + blk * p.CB, p.cand_idx + blk * p.CB,
                           p.cand_hist + blk * kBlockBins, p.cand_start + blk * kBlockBins,
                           wide ? final_hist(g) : nullptr);
          if (S.tid == 0) __stcg(p.cand_count + blk, n);
        }
      }
      if (nsplit > 1 && !to_rows) {
        // last piece of the group to finish merges the candidates of all pieces
        __threadfence();
        named_bar_sync(3, 256);
        if (epi == 0 && lane == 0) {
          const int prev = atomicAdd(p.done + I.sgroup, 1);
          misc->merge_flag = (prev == nsplit - 1);
        }
        named_bar_sync(3, 256);
        if (misc->merge_flag) {
          __threadfence();
          for (int g = g_first; g < I.gcount; g += 2) {
            const int64_t blk0 = (int64_t)I.cand_block + (int64_t)g * nsplit;
            PieceCut* pre = reinterpret_cast<PieceCut*>(misc->piece_pre) + (alt ? 0 : wg * (kMaxCtas + 1));
            merge_pieces(S, p, blk0, nsplit, smem_u32(ck_of(g)), smem_u32(ci_of(g)), hist_of(g),
                         &tok[g], pre, out_row(g), wide ? final_hist(g) : nullptr);
            named_bar_sync(S.bar, S.nt);  // the slot is free for the next row
          }
          if (wide)  // the shared histograms are empty again for the next layer
            for (int g = g_first; g < I.gcount; g += 2)
              for (int b = S.tid; b < kSharedHistWords; b += S.nt) __stcg(early_hist(g) + b, 0u);
          if (epi == 0 && lane == 0) p.done[I.sgroup] = 0;  // ready for the next layer
        }
      }
      named_bar_sync(3, 256);
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) raise_status(p.status, kStatusTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// Top-k of the rows a decode batch scored into the workspace: one CTA of
// 1024 threads per query row, an exact radix select over the row's keys held
// in shared memory.  The first level bins the scores linearly over the row's
// own value range (scores crowd into few exponent values, so bins by the top
// bits of the key would collide), emits every key above the bin holding the
// k-th largest and gathers that bin's keys, normally a few dozen, which are
// then ranked directly (one thread each; ties by position).  A cut bin of
// more than 1024 keys (heavily tied scores) is resolved instead by levels
// that bin the keys still in play by (key - lo) >> shift over their own key
// range [lo, hi]; keys all equal to lo = hi are taken in position order.  Key 0 marks a key that is not
// visible (bad page) and is never selected.
// ---------------------------------------------------------------------------
constexpr int kRowsThreads = 1024;
constexpr int kRowsBins = 2048;

struct RowsTopkParams {
  const uint32_t* score_rows;
  const int32_t* row_keys;   // keys of row t, 0 = not a workspace row
  int score_stride;
  int k;
  int32_t* topk;
};

struct RowsScratch {
  uint32_t hist[kRowsBins];
  uint32_t cand_key[1024];           // the first level's cut bin
  int32_t cand_pos[1024];
  uint32_t n_out, n_cand;            // warp-aggregated output and gather counters
  float vmin, vmax;
  uint32_t cut_lo, cut_hi;           // key range of the cut bin
  uint32_t warp_part[32];
  uint32_t lo, hi;           // key range of the level
  int cut_bin, above, total;
  int base;                  // outputs written so far
};

// Warp-aggregated slot in a shared counter for every lane whose flag is set
// (all 32 lanes call it).
__device__ __forceinline__ uint32_t warp_take(bool flag, uint32_t* counter) {
  const uint32_t m = __ballot_sync(0xffffffffu, flag);
  uint32_t base = 0;
  if ((threadIdx.x & 31) == 0 && m) base = atomicAdd(counter, (uint32_t)__popc(m));
  base = __shfl_sync(0xffffffffu, base, 0);
  uint32_t lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
  return base + (uint32_t)__popc(m & lt);
}

__host__ __device__ inline size_t rows_topk_smem(int score_stride) {
  return (size_t)score_stride * 4 + sizeof(RowsScratch) + 64;
}

// Exclusive block-wide prefix sum of one count per thread; *total = the sum.
__device__ __forceinline__ uint32_t rows_scan(uint32_t v, RowsScratch* sc, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sc->warp_part[warp] = x;
  __syncthreads();
  constexpr int kWarps = kRowsThreads / 32;
  if (warp == 0) {
    uint32_t w = lane < kWarps ? sc->warp_part[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) sc->warp_part[lane] = w;  // inclusive
  }
  __syncthreads();
  *total = sc->warp_part[kWarps - 1];
  const uint32_t ex = (warp > 0 ? sc->warp_part[warp - 1] : 0u) + x - v;
  __syncthreads();
  return ex;
}

// The bin holding the need-th largest key of sc->hist (bins from the top;
// each thread owns kRowsBins / kRowsThreads of them): sets sc->cut_bin (-1 when the bins hold at most
// `need` keys), sc->above (keys in higher bins) and sc->total (the bin's).
// Every thread calls it; it ends without a barrier.
__device__ __forceinline__ void rows_find_cut(RowsScratch* sc, int need);

// The score a key encodes (inverse of score_key).
__device__ __forceinline__ float key_score(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Shift that maps [lo, hi] onto at most kRowsBins bins: (key - lo) >> shift.
__device__ __forceinline__ int rows_shift(uint32_t lo, uint32_t hi) {
  const int bits = 32 - __clz(hi - lo);  // bit length of hi - lo
  return bits > 11 ? bits - 11 : 0;
}

__device__ __forceinline__ void rows_find_cut(RowsScratch* sc, int need) {
  constexpr int kPer = kRowsBins / kRowsThreads;
  const int tid = threadIdx.x;
  const int bt = kRowsBins - kPer * tid - 1;
  uint32_t cs[kPer], mine = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    cs[j] = sc->hist[bt - j];
    mine += cs[j];
  }
  uint32_t total;
  const uint32_t above = rows_scan(mine, sc, &total);
  if ((int)total <= need) {
    if (tid == 0) sc->cut_bin = -1;
  } else if ((int)above < need && need <= (int)(above + mine)) {
    uint32_t a = above;
    for (int j = 0; j < kPer; ++j) {
      if (need <= (int)(a + cs[j])) {
        sc->cut_bin = bt - j;
        sc->above = (int)a;
        sc->total = (int)cs[j];
        break;
      }
      a += cs[j];
    }
  }
}

__global__ void __launch_bounds__(kRowsThreads, 1) rows_topk_kernel(const __grid_constant__ RowsTopkParams p) {
  // launched while the scoring kernel runs; its keys are complete after this
  pdl_wait();
  const int t = blockIdx.x;
  extern __shared__ __align__(16) unsigned char rows_smem[];
  uint32_t* keys = reinterpret_cast<uint32_t*>(rows_smem);
  RowsScratch* sc = reinterpret_cast<RowsScratch*>(keys + p.score_stride);
  int32_t* out = p.topk + (int64_t)t * p.k;
  const int tid = threadIdx.x;
  // the whole row area to shared memory while the row's key count loads
  // (entries beyond it are not used)
  const uint32_t* row = p.score_rows + (int64_t)t * p.score_stride;
  const int n = __ldg(p.row_keys + t);
  for (int i = tid; i < p.score_stride; i += kRowsThreads) keys[i] = __ldcg(row + i);
  if (n <= 0) return;  // not a workspace row (uniform: every thread leaves)
  __syncthreads();
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  for (int i = tid; i < n; i += kRowsThreads) {
    const uint32_t kk = keys[i];
    if (kk != 0u) {
      kmin = min(kmin, kk);
      kmax = max(kmax, kk);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (tid == 0) { sc->lo = 0xFFFFFFFFu; sc->hi = 0u; sc->base = 0; }
  __syncthreads();
  if ((tid & 31) == 0) { atomicMin(&sc->lo, kmin); atomicMax(&sc->hi, kmax); }
  __syncthreads();
  uint32_t lo = sc->lo, hi = sc->hi;
  int need = p.k;
  bool done = lo > hi;  // no visible key
  if (!done) {
    // ---- first level: 2048 bins linear in the score over [vmin, vmax]
    const float vmin = key_score(lo), vmax = key_score(hi);
    const float scale = vmax > vmin ? (float)kRowsBins / (vmax - vmin) : 0.f;
    auto vbin = [&](uint32_t kk) -> int {  // monotone in the score
      const float b = (key_score(kk) - vmin) * scale;
      return b >= (float)(kRowsBins - 1) ? kRowsBins - 1 : (b > 0.f ? (int)b : 0);
    };
    for (int b = tid; b < kRowsBins; b += kRowsThreads) sc->hist[b] = 0u;
    if (tid == 0) { sc->cut_lo = 0xFFFFFFFFu; sc->cut_hi = 0u; }
    __syncthreads();
    for (int i = tid; i < n; i += kRowsThreads) {
      const uint32_t kk = keys[i];
      if (kk != 0u) atomicAdd(&sc->hist[vbin(kk)], 1u);
    }
    __syncthreads();
    rows_find_cut(sc, need);
    if (tid == 0) { sc->n_out = 0u; sc->n_cand = 0u; }
    __syncthreads();
    const int cut = sc->cut_bin;
    // emit the keys above the cut bin (every visible key when there is none)
    // and gather the cut bin's keys; positions from warp-aggregated counters
    // (the order inside the output row is free)
    uint32_t clo = 0xFFFFFFFFu, chi = 0u;
    for (int c0i = 0; c0i < n; c0i += kRowsThreads) {  // same bound for every thread
      const int i = c0i + tid;
      const uint32_t kk = i < n ? keys[i] : 0u;
      const int b = kk != 0u ? vbin(kk) : -2;
      const bool emit = kk != 0u && (cut < 0 || b > cut);
      const bool gather = kk != 0u && b == cut;
      const uint32_t po = warp_take(emit, &sc->n_out);
      if (emit) out[po] = i;
      const uint32_t pc = warp_take(gather, &sc->n_cand);
      if (gather) {
        if (pc < 1024u) {
          sc->cand_key[pc] = kk;
          sc->cand_pos[pc] = i;
        }
        clo = min(clo, kk);
        chi = max(chi, kk);
      }
    }
    __syncthreads();
    const uint32_t emitted = sc->n_out, m = sc->n_cand;
    if (cut < 0) {
      if (tid == 0) sc->base = (int)emitted;
      done = true;
    } else {
      need -= sc->above;
      if (m <= 1024u) {
        // rank of each gathered candidate: larger keys first, ties by position
        for (int j = tid; j < (int)m; j += kRowsThreads) {
          const uint32_t kj = sc->cand_key[j];
          const int pj = sc->cand_pos[j];
          int rank = 0;
          for (int i = 0; i < (int)m; ++i) {
            const uint32_t ki = sc->cand_key[i];
            rank += (ki > kj || (ki == kj && sc->cand_pos[i] < pj)) ? 1 : 0;
          }
          if (rank < need) out[emitted + rank] = pj;
        }
        if (tid == 0) sc->base = (int)emitted + min((int)m, need);
        done = true;
      } else {
        // heavily tied: resolve the cut bin by key-range levels
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          clo = min(clo, __shfl_xor_sync(0xffffffffu, clo, o));
          chi = max(chi, __shfl_xor_sync(0xffffffffu, chi, o));
        }
        if ((tid & 31) == 0) { atomicMin(&sc->cut_lo, clo); atomicMax(&sc->cut_hi, chi); }
        if (tid == 0) sc->base = (int)emitted;
        __syncthreads();
        lo = sc->cut_lo;
        hi = sc->cut_hi;
        if (lo == hi) {
          // every key of the cut bin is equal: the first `need` in position order
          const int per = (n + kRowsThreads - 1) / kRowsThreads;
          uint32_t eq = 0;
          for (int i = tid * per, e = 0; e < per && i < n; ++i, ++e) eq += keys[i] == lo ? 1u : 0u;
          const uint32_t base1 = (uint32_t)sc->base;
          uint32_t all;
          uint32_t rank = rows_scan(eq, sc, &all);
          uint32_t w = base1 + rank;
          for (int i = tid * per, e = 0; e < per && i < n; ++i, ++e)
            if (keys[i] == lo) {
              if (rank < (uint32_t)need) out[w] = i;
              ++rank;
              ++w;
            }
          __syncthreads();
          if (tid == 0) sc->base += min((int)all, need);
          done = true;
        }
      }
    }
    __syncthreads();
  }
  while (!done) {
    const int sh = rows_shift(lo, hi);
    // keys in play: lo <= key <= hi; count them per bin
    for (int b = tid; b < kRowsBins; b += kRowsThreads) sc->hist[b] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kRowsThreads) {
      const uint32_t kk = keys[i];
      if (kk != 0u && kk >= lo && kk <= hi) atomicAdd(&sc->hist[(kk - lo) >> sh], 1u);
    }
    __syncthreads();
    rows_find_cut(sc, need);
    __syncthreads();
    const int cut = sc->cut_bin;
    // emit the keys above the cut bin (all keys in play when there is no cut)
    const uint32_t base0 = (uint32_t)sc->base;  // thread 0 updates it after the scan's barriers
    uint32_t mine = 0;
    for (int i = tid; i < n; i += kRowsThreads) {
      const uint32_t kk = keys[i];
      mine += (kk != 0u && kk >= lo && kk <= hi && (cut < 0 || (int)((kk - lo) >> sh) > cut)) ? 1u : 0u;
    }
    uint32_t emitted;
    uint32_t pos = base0 + rows_scan(mine, sc, &emitted);
    for (int i = tid; i < n; i += kRowsThreads) {
      const uint32_t kk = keys[i];
      if (kk != 0u && kk >= lo && kk <= hi && (cut < 0 || (int)((kk - lo) >> sh) > cut)) out[pos++] = i;
    }
    if (cut < 0) {
      if (tid == 0) sc->base += (int)emitted;
      done = true;
    } else {
      need -= sc->above;
      // the cut bin's key range
      const uint32_t nlo = lo + ((uint32_t)cut << sh);
      const uint32_t nhi = (uint32_t)min((uint64_t)hi, (uint64_t)nlo + ((uint64_t)1 << sh) - 1u);
      if (tid == 0) sc->base += (int)emitted;
      lo = nlo;
      hi = nhi;
      if (lo == hi) {
        // every remaining key equals lo: the first `need` in position order
        __syncthreads();
        uint32_t eq = 0;
        for (int i = tid * ((n + kRowsThreads - 1) / kRowsThreads), e = 0;
             e < (n + kRowsThreads - 1) / kRowsThreads && i < n; ++i, ++e)
          eq += keys[i] == lo ? 1u : 0u;
        const uint32_t base1 = (uint32_t)sc->base;
        uint32_t all;
        uint32_t rank = rows_scan(eq, sc, &all);
        uint32_t w = base1 + rank;
        for (int i = tid * ((n + kRowsThreads - 1) / kRowsThreads), e = 0;
             e < (n + kRowsThreads - 1) / kRowsThreads && i < n; ++i, ++e)
          if (keys[i] == lo) {
            if (rank < (uint32_t)need) out[w] = i;
            ++rank;
            ++w;
          }
        __syncthreads();
        if (tid == 0) sc->base += min((int)all, need);
        done = true;
      }
    }
    __syncthreads();
  }
  // -1 after the selected keys
  const int filled = sc->base;
  for (int i = filled + tid; i < p.k; i += kRowsThreads) out[i] = -1;
}

}  // namespace dsa
