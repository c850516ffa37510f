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
//   warp 0      producer: per key tile (128 keys = 2 pages) two TMA loads of
//               64 x 128 B key rows into a 128B-swizzled stage plus two 256 B
//               bulk copies of the pages' scales; the query tile of each item
//               (double-buffered when it is small).
//   warp 1      owns tensor memory; one lane issues 4 tcgen05.mma (K = 32
//               each) per tile: D[key, row*H + head] += k . q, FP32 in TMEM.
//   warps 2-9   epilogue, two warpgroups; thread = one key row of the tile
//               (its TMEM lane).  For each query row of the group: read the
//               H accumulators, ReLU, weight, sum, times the key's scale,
//               then stream the score into an exact top-k buffer in shared
//               memory (append above the running threshold; when the buffer
//               fills, radix-select the k largest and raise the threshold).
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
constexpr int kMaxStages = 16;
constexpr int kMaxAccBufs = 8;
constexpr int kMaxQBufs = 2;
constexpr int kTmemCols = 512;
constexpr int kMergePer = 4;              // candidates per thread per merge batch

struct TokSlot {
  int32_t count;   // candidates held
  uint32_t thr;    // keys <= thr are not admitted
  int32_t pos;     // position of the query row in its request
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
  int T, H, G, k, C, NS, NB, NQ, n_max;
  int q_box_per_token;
  uint32_t q_bytes;  // bytes of one query-tile buffer
  const Item* items;
  const PlanHeader* hdr;
  uint32_t* cand_keys;
  int32_t* cand_idx;
  int32_t* cand_count;
  int32_t* done;
  int32_t* topk;
  float* scores_out;
  int64_t scores_ld;
  int32_t* status;
  // dynamic shared memory offsets (from a 1024-aligned base)
  uint32_t off_stage, off_q, off_ckeys, off_cidx, off_wq, off_tok, off_hist, off_misc, off_bar;
};

struct SelScratch {
  int scan[8];                 // per-warp partials of a block scan (up to 256 threads)
  int bin, above, cnt;
  uint32_t lo, hi;
  int pad[3];
};

struct Misc {
  int abort;       // any role gave up (producer and MMA stop early on it)
  uint32_t tmem_base;
  int merge_flag;
  int epi_abort;   // an epilogue wait gave up; read by the epilogue only after barriers
  SelScratch sel[2];
};

// The candidates of one query row are selected by a "selector": either one
// warpgroup (128 threads, its own rows) or both (256 threads, the single row
// of a decode item).  A selector names its threads, its named barrier and its
// scratch.
struct Selector {
  int nt;          // threads
  int tid;         // this thread, 0..nt-1
  uint32_t bar;    // named barrier id
  int* unused;
  SelScratch* s;
};

constexpr int kSelRegs = 32;   // candidates a selector thread holds in registers
constexpr int kBins = 2048;

struct Thresh {
  uint32_t prefix;  // keys >= prefix are taken (early), or > prefix plus `need` ties (exact)
  int need;
  int early;
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan of one int per selector thread; *total gets the sum.
__device__ __forceinline__ int sel_scan(const Selector S, int v, int* total) {
  const int lane = S.tid & 31, w = S.tid >> 5, nw = S.nt >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) S.s->scan[w] = x;
  named_bar_sync(S.bar, S.nt);
  int off = 0, tot = 0;
  for (int u = 0; u < nw; ++u) {
    const int c = S.s->scan[u];
    if (u < w) off += c;
    tot += c;
  }
  named_bar_sync(S.bar, S.nt);
  *total = tot;
  return off + x - v;
}

constexpr int kHistShift = 21;  // level-1 bin of a key: its top 11 bits (sign, exponent, 2 mantissa)

struct BinCut {
  int bin;    // the bin holding the need-th largest key
  int above;  // keys in higher bins
  int cnt;    // keys in that bin
};

// Walk a 2048-bin histogram (shared memory) from the top; find the bin where
// the running count reaches `need`.  Every selector thread gets the result.
__device__ __forceinline__ BinCut find_bin(const Selector S, uint32_t hist_s, int need) {
  const int per = kBins / S.nt;               // 8 or 16 bins per thread, highest first
  const int top = kBins - 1 - S.tid * per;
  uint32_t hv[kBins / 128];
#pragma unroll
  for (int j = 0; j < kBins / 128; ++j) hv[j] = lds_u32_if(j < per, hist_s + 4 * (top - j));
  int local = 0;
#pragma unroll
  for (int j = 0; j < kBins / 128; ++j) local += (int)hv[j];
  int total;
  int above = sel_scan(S, local, &total);
  if (above < need && need <= above + local) {
    for (int j = 0; j < per; ++j) {
      const int c = (int)hv[j];
      if (need <= above + c) {
        S.s->bin = top - j;
        S.s->above = above;
        S.s->cnt = c;
        break;
      }
      above += c;
    }
  }
  named_bar_sync(S.bar, S.nt);
  const BinCut r{S.s->bin, S.s->above, S.s->cnt};
  named_bar_sync(S.bar, S.nt);
  return r;
}

// Exact threshold of the k-th largest register-held key, starting from the
// level-1 bin cut `c` (taken from the incremental histogram): refine inside
// that bin on key bits 20..10, then 9..0, using scratch_s (2048 ints of
// shared memory) for the sub-histograms.  Stops as soon as a whole sub-bin is
// taken.
__device__ __forceinline__ Thresh refine_in_bin(const Selector S, const uint32_t* kr, BinCut c,
                                                int k, uint32_t scratch_s) {
  Thresh th{(uint32_t)c.bin << kHistShift, k - c.above, 0};
  uint32_t mask = 0xFFFFFFFFu << kHistShift;
  if (c.cnt == th.need) {
    th.early = 1;
    return th;
  }
  for (int level = 0; level < 2; ++level) {
    const int shift = level == 0 ? 10 : 0;
    const uint32_t dm = level == 0 ? 2047u : 1023u;
    for (int b = S.tid; b < kBins; b += S.nt) sts_u32(scratch_s + 4 * b, 0u);
    named_bar_sync(S.bar, S.nt);
#pragma unroll
    for (int j = 0; j < kSelRegs; ++j)
      red_add_shared_if(kr[j] != 0u && (kr[j] & mask) == th.prefix,
                        scratch_s + 4 * ((kr[j] >> shift) & dm), 1u);
    named_bar_sync(S.bar, S.nt);
    const BinCut c2 = find_bin(S, scratch_s, th.need);
    th.need -= c2.above;
    th.prefix |= (uint32_t)c2.bin << shift;
    mask |= dm << shift;
    if (c2.cnt == th.need) {
      th.early = 1;
      break;
    }
  }
  return th;
}

// Write the selected keys (th) of the selector's registers kr (with their
// indices from idx_src[tid + nt*j]) to dkeys/didx[0, ...), in (thread,
// register) order: deterministic.  Ties at an exact threshold are taken in
// that order up to the quota.  dst may alias the source buffers (everything is
// read before anything is written).  Returns the number written.
__device__ __forceinline__ int compact_selected(const Selector S, const uint32_t* kr,
                                                const int32_t* idx_src, Thresh th,
                                                uint32_t* dkeys, int32_t* didx) {
  int nsel = 0, ntie = 0;
#pragma unroll
  for (int j = 0; j < kSelRegs; ++j) {
    const uint32_t key = kr[j];
    nsel += (key != 0u && (th.early ? key >= th.prefix : key > th.prefix)) ? 1 : 0;
    ntie += (key != 0u && !th.early && key == th.prefix) ? 1 : 0;
  }
  int tie_tot;
  const int tie_off = sel_scan(S, ntie, &tie_tot);
  const int quota = th.early ? 0 : th.need;
  int take = quota - tie_off;
  take = take < 0 ? 0 : (take > ntie ? ntie : take);
  int total;
  int pos = sel_scan(S, nsel + take, &total);
  int32_t ix[kSelRegs];
  const uint32_t ia = smem_u32(idx_src);
#pragma unroll
  for (int j = 0; j < kSelRegs; ++j) ix[j] = (int32_t)lds_u32_if(kr[j] != 0u, ia + 4 * (S.tid + S.nt * j));
  named_bar_sync(S.bar, S.nt);  // every source index is read before any write
  int ties = 0;
#pragma unroll
  for (int j = 0; j < kSelRegs; ++j) {
    const uint32_t key = kr[j];
    const bool above = key != 0u && (th.early ? key >= th.prefix : key > th.prefix);
    const bool tie = key != 0u && !th.early && key == th.prefix && ties < take;
    ties += tie ? 1 : 0;
    if (above || tie) {
      if (dkeys) dkeys[pos] = key;
      didx[pos] = ix[j];
      ++pos;
    }
  }
  named_bar_sync(S.bar, S.nt);
  return total;
}

__device__ __forceinline__ void load_regs(const Selector S, const uint32_t* ck, int n,
                                          uint32_t* kr) {
  const uint32_t a = smem_u32(ck);
#pragma unroll
  for (int j = 0; j < kSelRegs; ++j) {
    const int i = S.tid + S.nt * j;
    kr[j] = lds_u32_if(i < n, a + 4 * i);
  }
}

__device__ __forceinline__ void hist_clear(const Selector S, uint32_t hist_s) {
  for (int b = S.tid; b < kBins; b += S.nt) sts_u32(hist_s + 4 * b, 0u);
}

// Shrink a slot's buffer while streaming: keep every candidate in or above the
// level-1 bin of the k-th largest (at least k, usually a little more), zero
// the histogram below it and raise the admission threshold to that bin's lower
// edge.  If that bin alone would not leave `limit` room, select exactly k.
__device__ __noinline__ void slot_compress(const Selector S, TokSlot* ts, uint32_t* ck,
                                           int32_t* ci, uint32_t hist_s, int k, int limit) {
  uint32_t kr[kSelRegs];
  const int n = ts->count;
  load_regs(S, ck, n, kr);
  const BinCut c = find_bin(S, hist_s, k);
  if (c.above + c.cnt <= limit) {
    const Thresh th{(uint32_t)c.bin << kHistShift, 0, 1};
    const int kept = compact_selected(S, kr, ci, th, ck, ci);
    const int per = kBins / S.nt;
    const int top = kBins - 1 - S.tid * per;
    for (int j = 0; j < per; ++j)
      if (top - j < c.bin) sts_u32(hist_s + 4 * (top - j), 0u);
    if (S.tid == 0) {
      ts->count = kept;
      ts->thr = th.prefix > 0u ? th.prefix - 1u : 0u;
    }
  } else {
    const Thresh th = refine_in_bin(S, kr, c, k, hist_s);
    const int kept = compact_selected(S, kr, ci, th, ck, ci);
    // rebuild the histogram of what is kept
    hist_clear(S, hist_s);
    named_bar_sync(S.bar, S.nt);
    load_regs(S, ck, kept, kr);
#pragma unroll
    for (int j = 0; j < kSelRegs; ++j)
      red_add_shared_if(kr[j] != 0u, hist_s + 4 * (kr[j] >> kHistShift), 1u);
    if (S.tid == 0) {
      ts->count = kept;
      ts->thr = th.early ? (th.prefix > 0u ? th.prefix - 1u : 0u) : th.prefix;
    }
  }
  named_bar_sync(S.bar, S.nt);
}

// Final selection of a slot: write its min(count, k) largest candidates
// (keys to dkeys unless null, indices to didx).  The slot's histogram serves
// as scratch and is left undefined.  Returns how many were written.
__device__ __noinline__ int slot_emit(const Selector S, TokSlot* ts, const uint32_t* ck,
                                      const int32_t* ci, uint32_t hist_s, int k, uint32_t* dkeys,
                                      int32_t* didx) {
  uint32_t kr[kSelRegs];
  const int n = ts->count;
  load_regs(S, ck, n, kr);
  Thresh th{0u, 0, 1};  // everything
  if (n > k) th = refine_in_bin(S, kr, find_bin(S, hist_s, k), k, hist_s);
  return compact_selected(S, kr, ci, th, dkeys, didx);
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

template <int H>
__device__ __forceinline__ float relu_weighted_sum(uint32_t taddr, const float* wq) {
  constexpr int CH = H >= 32 ? 32 : H;              // columns per tcgen05.ld
  constexpr int BATCH = H >= 64 ? 64 : H;           // columns loaded before one wait
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int c0 = 0; c0 < H; c0 += BATCH) {
    uint32_t v[BATCH];
#pragma unroll
    for (int c = 0; c < BATCH; c += CH) tmem_ld<CH>(taddr + c0 + c, v + c);
    tmem_ld_wait();
    const float4* w4 = reinterpret_cast<const float4*>(wq + c0);
#pragma unroll
    for (int h = 0; h < BATCH; h += 4) {
      const float4 ww = w4[h >> 2];
      acc0 = fmaf(ww.x, fmaxf(__uint_as_float(v[h + 0]), 0.f), acc0);
      acc1 = fmaf(ww.y, fmaxf(__uint_as_float(v[h + 1]), 0.f), acc1);
      acc0 = fmaf(ww.z, fmaxf(__uint_as_float(v[h + 2]), 0.f), acc0);
      acc1 = fmaf(ww.w, fmaxf(__uint_as_float(v[h + 3]), 0.f), acc1);
    }
  }
  return acc0 + acc1;
}

template <int H>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_topk_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_q, const ScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  // align to 1024 by pointer arithmetic on the shared array itself, so the
  // compiler keeps every access below in the shared address space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint8_t* stage_base = smem + p.off_stage;
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
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);  // freed by the MMA commit
    }
    for (int b = 0; b < p.NB; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      // decode layout: one warpgroup reads a tile; otherwise both do
      mbar_init(bar_tempty + 8 * b, p.G == 1 ? kEpiWarps / 2 : kEpiWarps);
    }
    for (int b = 0; b < p.NQ; ++b) {
      mbar_init(bar_qfull + 8 * b, 1);
      mbar_init(bar_qempty + 8 * b, 1);
    }
    mbar_init(bar_drain, 1);
    misc->abort = 0;
    misc->epi_abort = 0;
    misc->merge_flag = 0;
    for (int i = 0; i < 2; ++i) {
      misc->sel[i].lo = 0xFFFFFFFFu;
      misc->sel[i].hi = 0u;
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_q);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc->tmem_base;
  const int n_items = p.hdr->n_items;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the tiles; lane 0 waits and issues the two key-page
    // copies of each tile (each bulk-copy issue costs the thread ~100 cycles,
    // so nothing else is issued here).  The page ids of 16 tiles (32 pages)
    // come from one coalesced load, fetched one chunk ahead.
    int stage = 0;
    uint32_t sphase = 0;
    uint32_t issued_mask = 0;
    uint32_t last_par[kMaxStages];
    int q_last[kMaxQBufs] = {-1, -1};
    int item_i = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++item_i) {
      const Item I = p.items[it];
      const int qb = item_i % p.NQ;
      const uint32_t qpar = (uint32_t)((item_i / p.NQ) & 1);
      int okv = 1;
      if (lane == 0) okv = mbar_wait(bar_qempty + 8 * qb, qpar ^ 1, abort_flag);
      if (!__shfl_sync(0xffffffffu, okv, 0)) { ok = false; break; }
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
      const int ntiles = (I.k1 - I.k0 + kTileKeys - 1) / kTileKeys;
      const int32_t* bt_row = p.block_table + (int64_t)I.r * p.max_blocks;
      const int page0 = I.k0 / kPageTokens;
      auto load_pages = [&](int chunk) -> int64_t {  // this lane's page of a 32-page chunk
        const int pidx = page0 + chunk * 32 + lane;
        int64_t page = -1;
        if (chunk * 16 < ntiles && pidx * kPageTokens < I.k1) {
          page = __ldg(bt_row + pidx);
          if (page < 0 || page >= p.num_pages) page = -1;
        }
        return page;
      };
      int64_t cur = load_pages(0);
      for (int c = 0; c * 16 < ntiles && ok; ++c) {
        const int64_t nxt = load_pages(c + 1);
        const int jend = min(16, ntiles - c * 16);
        for (int jj = 0; jj < jend; ++jj) {
          const int64_t pg0 = __shfl_sync(0xffffffffu, cur, 2 * jj);
          const int64_t pg1 = __shfl_sync(0xffffffffu, cur, 2 * jj + 1);
          okv = 1;
          if (lane == 0) {
            okv = mbar_wait(bar_empty + 8 * stage, sphase ^ 1, abort_flag);
            if (okv) {
              const uint32_t bytes = (pg0 >= 0 ? kPageTokens * kHeadDim : 0) +
                                     (pg1 >= 0 ? kPageTokens * kHeadDim : 0);
              mbar_arrive_expect_tx(bar_full + 8 * stage, bytes);
              const uint32_t dst = smem_u32(stage_base + stage * kStageBytes);
              if (pg0 >= 0)
                tma_load_2d(dst, &tm_k, 0, (int32_t)(pg0 * (kPageBytes / kHeadDim)),
                            bar_full + 8 * stage);
              if (pg1 >= 0)
                tma_load_2d(dst + kPageTokens * kHeadDim, &tm_k, 0,
                            (int32_t)(pg1 * (kPageBytes / kHeadDim)), bar_full + 8 * stage);
            }
          }
          if (!__shfl_sync(0xffffffffu, okv, 0)) { ok = false; break; }
          issued_mask |= 1u << stage;
          last_par[stage] = sphase;
          if (++stage == p.NS) { stage = 0; sphase ^= 1; }
        }
        cur = nxt;
      }
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, kStatusTimeout);
      }
      // never leave with bulk copies in flight into this CTA's shared memory
      for (int s = 0; s < p.NS; ++s)
        if (issued_mask & (1u << s)) mbar_wait(bar_full + 8 * s, last_par[s], nullptr);
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
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++item_i) {
        const Item I = p.items[it];
        const uint32_t N = (uint32_t)((I.gcount * H + 15) & ~15);
        const uint32_t idesc = idesc_e4m3_f32(128, N);
        const int qb = item_i % p.NQ;
        if (!mbar_wait(bar_qfull + 8 * qb, (uint32_t)((item_i / p.NQ) & 1), abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t qaddr = smem_u32(q_base + qb * p.q_bytes);
        const int ntiles = (I.k1 - I.k0 + kTileKeys - 1) / kTileKeys;
        for (int j = 0; j < ntiles; ++j) {
          if (!mbar_wait(bar_full + 8 * stage, sphase, abort_flag)) { ok = false; break; }
          if (!mbar_wait(bar_tempty + 8 * acc, aphase ^ 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t aaddr = smem_u32(stage_base + stage * kStageBytes);
          const uint32_t d = tmem_base + (uint32_t)(acc * p.n_max);
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 32; ++kk)
            umma_f8(d, sw128_desc(aaddr + kk * 32), sw128_desc(qaddr + kk * 32), idesc, kk > 0);
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
    // the group and both read every tile.  Each thread fetches its key's scale
    // and page id itself, a few tiles ahead of use.
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
    // buffer-fill checks every `chk` iterations, leaving room for what they append
    const int chk = alt ? 8 : 4;
    const int headroom = chk * kTileKeys * (alt ? 2 : 1);
    long long tile_base = 0;  // tiles of earlier items of this CTA (all roles count alike)
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const Item I = p.items[it];
      const int qb0 = __ldg(p.qsl + I.r);
      const int q_len = __ldg(p.qsl + I.r + 1) - qb0;
      const int seq_len = __ldg(p.seq_lens + I.r);
      const int nsplit = I.split >> 16;
      const int split = I.split & 0xFFFF;
      const int g_first = alt ? 0 : wg;  // this thread's rows: g_first, g_first + 2, ...
      // per-row setup (warpgroup 0 for the shared decode row)
      for (int g = g_first; g < I.gcount; g += 2) {
        const int t = I.t0 + g;
        if (!alt || wg == 0) {
          for (int h = tid; h < H; h += 128)
            wq_all[g * H + h] =
                __ldg(p.w + (int64_t)t * H + h) * __ldg(p.q_scale + (int64_t)t * H + h);
          if (tid == 0) {
            tok[g].count = 0;
            tok[g].thr = 0u;
            tok[g].pos = seq_len - q_len + (t - qb0);
            tok[g].t = t;
          }
        }
      }
      for (int g = g_first; g < I.gcount; g += 2) hist_clear(S, hist_of(g));
      named_bar_sync(3, 256);
      const int ntiles = (I.k1 - I.k0 + kTileKeys - 1) / kTileKeys;
      const bool may_fill = (I.k1 - I.k0) > p.C;
      const int32_t* bt_row = p.block_table + (int64_t)I.r * p.max_blocks;
      auto page_of = [&](int jj) -> int64_t {  // -1: beyond the range, -2: invalid id
        const int key = I.k0 + jj * kTileKeys + row;
        if (jj >= ntiles || key >= I.k1) return -1;
        const int64_t pg = __ldg(bt_row + key / kPageTokens);
        return (pg >= 0 && pg < p.num_pages) ? pg : -2;
      };
      auto scale_of = [&](int64_t pg, int jj) -> float {
        if (pg < 0) return 0.f;
        const int key = I.k0 + jj * kTileKeys + row;
        return __ldg(reinterpret_cast<const float*>(p.k_cache + pg * kPageBytes +
                                                    kPageScaleOffset) + (key % kPageTokens));
      };
      const int j0 = alt ? wg : 0;
      int64_t pg0 = page_of(j0), pg1 = page_of(j0 + step), pg2 = page_of(j0 + 2 * step),
              pg3 = page_of(j0 + 3 * step), pg4 = page_of(j0 + 4 * step);
      float sc0 = scale_of(pg0, j0), sc1 = scale_of(pg1, j0 + step), sc2 = scale_of(pg2, j0 + 2 * step);
      const int iters = alt ? (ntiles + 1) / 2 : ntiles;
      for (int m = 0; m < iters; ++m) {
        const int j = j0 + m * step;
        // prefetch: scale three own tiles ahead, page id five ahead
        const float sc3 = scale_of(pg3, j + 3 * step);
        const int64_t pg5 = page_of(j + 5 * step);
        if (j < ntiles && ok) {
          const long long seq = tile_base + j;
          const int acc = (int)(seq % p.NB);
          const uint32_t aphase = (uint32_t)((seq / p.NB) & 1);
          const int key = I.k0 + j * kTileKeys + row;
          const bool kvalid = pg0 >= 0;
          if (pg0 == -2 && lane == 0) raise_status(p.status, kStatusBadPage);
          // no early exit on the abort flag here: the warps of a warpgroup must take
          // the same branch, so they all wait on the same phase with the same limit
          if (!mbar_wait(bar_tfull + 8 * acc, aphase, nullptr)) ok = false;
          if (ok) {
            tc_fence_after();
            const uint32_t tbase =
                tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * p.n_max);
            for (int g = g_first; g < I.gcount; g += 2) {
              const float s = relu_weighted_sum<H>(tbase + (uint32_t)(g * H), wq_all + g * H);
              const float score = s * sc0;
              const bool valid = kvalid && key <= tok[g].pos;
              if (p.scores_out && valid && key < p.scores_ld)
                p.scores_out[(int64_t)tok[g].t * p.scores_ld + key] = score;
              const uint32_t kk = valid ? score_key(score) : 0u;
              slot_append(kk, key, tok[g].thr, &tok[g], ckeys_all + (size_t)g * p.C,
                          cidx_all + (size_t)g * p.C, hist_of(g));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
          }
        }
        if (may_fill && (m % chk) == chk - 1 && m + 1 < iters) {
          if (!ok) misc->epi_abort = 1;
          named_bar_sync(3, 256);  // every append so far is visible
          if (misc->epi_abort) {
            ok = false;
          } else {
            for (int g = g_first; g < I.gcount; g += 2)
              if (tok[g].count > p.C - headroom)
                slot_compress(S, &tok[g], ckeys_all + (size_t)g * p.C, cidx_all + (size_t)g * p.C,
                              hist_of(g), p.k, p.C - headroom);
          }
          named_bar_sync(3, 256);
        }
        pg0 = pg1; pg1 = pg2; pg2 = pg3; pg3 = pg4; pg4 = pg5;
        sc0 = sc1; sc1 = sc2; sc2 = sc3;
      }
      tile_base += ntiles;
      if (!ok) misc->epi_abort = 1;
      named_bar_sync(3, 256);  // every append of the item is done
      if (misc->epi_abort) { ok = false; break; }
      // finalize this item's rows
      for (int g = g_first; g < I.gcount; g += 2) {
        uint32_t* ck = ckeys_all + (size_t)g * p.C;
        int32_t* ci = cidx_all + (size_t)g * p.C;
        if (nsplit == 1) {
          int32_t* out_row = p.topk + (int64_t)tok[g].t * p.k;
          const int n = slot_emit(S, &tok[g], ck, ci, hist_of(g), p.k, nullptr, out_row);
          for (int i = n + S.tid; i < p.k; i += S.nt) out_row[i] = -1;
        } else {
          const int64_t blk = (int64_t)I.cand_block + (int64_t)g * nsplit + split;
          const int n = slot_emit(S, &tok[g], ck, ci, hist_of(g), p.k, p.cand_keys + blk * p.k,
                                  p.cand_idx + blk * p.k);
          if (S.tid == 0) p.cand_count[blk] = n;
        }
      }
      if (nsplit > 1) {
        // last split of the group to finish merges the candidates of all splits
        __threadfence();
        named_bar_sync(3, 256);
        if (epi == 0 && lane == 0) {
          const int prev = atomicAdd(p.done + I.sgroup, 1);
          misc->merge_flag = (prev == nsplit - 1);
        }
        named_bar_sync(3, 256);
        if (misc->merge_flag) {
          __threadfence();
          const int batch = S.nt * kMergePer;
          for (int g = g_first; g < I.gcount; g += 2) {
            uint32_t* ck = ckeys_all + (size_t)g * p.C;
            int32_t* ci = cidx_all + (size_t)g * p.C;
            if (S.tid == 0) {
              tok[g].count = 0;
              tok[g].thr = 0u;
            }
            hist_clear(S, hist_of(g));
            named_bar_sync(S.bar, S.nt);
            for (int sj = 0; sj < nsplit; ++sj) {
              const int64_t blk = (int64_t)I.cand_block + (int64_t)g * nsplit + sj;
              const int nb = __ldcg(p.cand_count + blk);
              const uint32_t* gk = p.cand_keys + blk * p.k;
              const int32_t* gi = p.cand_idx + blk * p.k;
              for (int i0 = 0; i0 < nb; i0 += batch) {
                uint32_t kk[kMergePer];
                int32_t ix[kMergePer];
#pragma unroll
                for (int u = 0; u < kMergePer; ++u) {
                  const int i = i0 + u * S.nt + S.tid;
                  kk[u] = (i < nb) ? __ldcg(gk + i) : 0u;
                  ix[u] = (i < nb) ? __ldcg(gi + i) : -1;
                }
                const uint32_t thr = tok[g].thr;
#pragma unroll
                for (int u = 0; u < kMergePer; ++u)
                  slot_append(kk[u], ix[u], thr, &tok[g], ck, ci, hist_of(g));
                named_bar_sync(S.bar, S.nt);
                if (tok[g].count > p.C - batch)
                  slot_compress(S, &tok[g], ck, ci, hist_of(g), p.k, p.C - batch);
              }
            }
            int32_t* out_row = p.topk + (int64_t)tok[g].t * p.k;
            const int n = slot_emit(S, &tok[g], ck, ci, hist_of(g), p.k, nullptr, out_row);
            for (int i = n + S.tid; i < p.k; i += S.nt) out_row[i] = -1;
          }
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

}  // namespace dsa
