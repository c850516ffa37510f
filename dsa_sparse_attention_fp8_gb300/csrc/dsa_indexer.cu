// C ABI of the DSA lightning-indexer library: argument checks, launch
// configuration, tensor-map encoding and kernel launches.  See
// include/dsa_indexer.h for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "dsa_indexer.h"
#include "kwrite.cuh"
#include "mla.cuh"
#include "plan.cuh"
#include "score_topk.cuh"

namespace {

thread_local std::string g_last_error;
thread_local int g_last_launches = 0;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return DSA_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// CTAs of the scoring launch: one per SM, at most kMaxCtas.  Without a
// device (sizing only) the bound itself is used, which over-sizes safely.
int grid_ctas() {
  const int n = sm_count();
  if (n <= 0 || n > dsa::kMaxCtas) return dsa::kMaxCtas;
  return n;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_heads(int H) {
  return H == 4 || H == 8 || H == 16 || H == 32 || H == 64 || H == 128;
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D uint8 view [rows, 128] with a box of `box_rows` x 128 bytes, 128-byte
// swizzle (or none).
int make_rows128_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows,
                     bool swizzle = true) {
  auto fn = encode_fn();
  if (!fn) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DSA_OK;
}

// Tuning overrides read from the environment: DSA_MIN_SPLIT (keys, the
// smallest per-CTA share of key tiles worth a piece of its own, default 1024),
// DSA_STAGE_KEYS (128 or 256, the decode layout's keys per pipeline stage,
// default 256), DSA_GROUP_ROWS (cap on query rows per group), DSA_PDL (0
// turns off programmatic dependent launch of the scoring kernel) and
// DSA_WAIT_LIMIT (iterations a scoring-kernel wait on another role may take,
// default and maximum kWaitLimit; 0 makes every such wait give up at once, to
// exercise the timeout path: the call then reports DSA_STATUS_TIMEOUT).
int env_int(const char* name, int dflt, int lo, int hi) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  const int x = atoi(v);
  return x < lo ? lo : (x > hi ? hi : x);
}

// ---------------------------------------------------------------- launch shape
struct ScoreShape {
  int G, C, NS, NB, NQ, NR, BPS, n_max, q_box_per_token;
  int lg_nb, lg_nr, lg_bps;
  uint32_t q_bytes;
  size_t smem_bytes;
  dsa::ScoreParams offs;  // only the off_* fields are filled
};

constexpr size_t kSmemLimit = 232448;  // 227 KB opt-in per block on sm_100-family

// Shared memory for the rows' candidate buffers and histograms of a group.
constexpr int kRowBudget = 128 * 1024;

// Candidate-buffer capacity per query row: at least k plus room for the
// candidates appended between two fill checks, and as much more as the rows'
// budget allows (up to 8192), so that rows shrink their buffer rarely.  A
// decode layout (one row per group) takes 6144, which leaves room for four
// 256-key pipeline stages.
int candidate_capacity(int k, int G, bool decode) {
  if (decode) return std::max(6144, (k + 1024 + 127) / 128 * 128);
  int c = ((kRowBudget / G - dsa::kBins * 4) / 8) / 128 * 128;
  c = std::min(c, 8192);
  return std::max(c, (k + 1024 + 127) / 128 * 128);
}

// Rows per group: one row per decode batch (no request has more rows than
// one), else as many rows as fill N = 128 of the MMA while each row's
// minimal candidate buffer and histogram fit the rows' budget.  Two rows of
// 64 heads with 7K-candidate buffers measured faster than four with 3K
// (fewer buffer shrinks outweigh the second read of each key tile, which
// hits L2).  DSA_GROUP_ROWS lowers it further.
int choose_group(int T, int R, int H, int k) {
  if (T <= R) return 1;
  int g = H >= 128 ? 1 : 128 / H;
  const int per_row = ((k + 1024 + 127) / 128 * 128) * 8 + dsa::kBins * 4;
  const int by_smem = kRowBudget / per_row;
  if (g > by_smem) g = by_smem;
  g = std::min(g, env_int("DSA_GROUP_ROWS", g, 1, 256));
  return g < 1 ? 1 : g;
}

size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int floor_log2(int x) {
  int l = 0;
  while ((2 << l) <= x) ++l;
  return l;
}

bool score_shape(int T, int R, int H, int k, ScoreShape* s) {
  s->G = choose_group(T, R, H, k);
  s->C = candidate_capacity(k, s->G, s->G == 1);
  s->q_box_per_token = (H % 8 == 0) ? 1 : 0;
  s->n_max = (s->G * H + 15) / 16 * 16;
  // decode layout: 256-key stages (two 128-key MMA blocks) when tensor memory
  // still holds 4 stage accumulators; halves the per-key barrier and issue work
  s->BPS = (s->G == 1 && dsa::kTmemCols / (2 * s->n_max) >= 4) ? 2 : 1;
  if (env_int("DSA_STAGE_KEYS", 256, 128, 256) < 256) s->BPS = 1;
  s->lg_bps = s->BPS == 2 ? 1 : 0;
  // accumulator buffers: a power of two, so the kernel's ring positions are masks
  s->NB = std::min(dsa::kTmemCols / (s->BPS * s->n_max), dsa::kMaxAccBufs);
  if (s->NB < 2) return false;
  s->lg_nb = floor_log2(s->NB);
  s->NB = 1 << s->lg_nb;
  s->q_bytes = (uint32_t)up((size_t)s->G * H * 128, 1024);
  s->NQ = s->q_bytes <= 16384 ? 2 : 1;
  size_t fixed = 0;
  fixed += (size_t)s->NQ * s->q_bytes;
  fixed += up((size_t)s->G * s->C * 4, 16) * 2;
  fixed += up((size_t)s->G * H * 4, 16);
  fixed += up((size_t)s->G * sizeof(dsa::TokSlot), 16);
  fixed += (size_t)s->G * dsa::kBins * 4;
  fixed += up(sizeof(dsa::Misc), 16);
  fixed += (2 * dsa::kMaxStages + 2 * dsa::kMaxAccBufs + 2 * dsa::kMaxQBufs + 1) * 8;
  const size_t stage_bytes = (size_t)s->BPS * dsa::kStageBytes;
  const size_t slot_bytes = (size_t)s->BPS * dsa::kScaleSlotBytes;
  const size_t budget = kSmemLimit - 1024 - 64;
  // stages, and a scale ring of NR >= NS + NB slots, NR a power of two
  auto ring = [&](int ns) { return 1 << floor_log2(2 * (ns + s->NB) - 1); };
  int ns = dsa::kMaxStages;
  while (ns >= 2 && fixed + ns * stage_bytes + ring(ns) * slot_bytes > budget) --ns;
  if (ns < 2) return false;
  s->NS = ns;
  s->NR = ring(ns);
  s->lg_nr = floor_log2(s->NR);
  size_t o = 0;  // stages first: every key stage starts on a 1024-byte boundary
  s->offs.off_stage = (uint32_t)o; o += (size_t)s->NS * stage_bytes;
  s->offs.off_scale = (uint32_t)o; o += (size_t)s->NR * slot_bytes;
  s->offs.off_q = (uint32_t)o;     o += (size_t)s->NQ * s->q_bytes;
  s->offs.off_ckeys = (uint32_t)o; o += up((size_t)s->G * s->C * 4, 16);
  s->offs.off_cidx = (uint32_t)o;  o += up((size_t)s->G * s->C * 4, 16);
  s->offs.off_wq = (uint32_t)o;    o += up((size_t)s->G * H * 4, 16);
  s->offs.off_tok = (uint32_t)o;   o += up((size_t)s->G * sizeof(dsa::TokSlot), 16);
  s->offs.off_hist = (uint32_t)o;  o += (size_t)s->G * dsa::kBins * 4;
  s->offs.off_misc = (uint32_t)o;  o += up(sizeof(dsa::Misc), 16);
  s->offs.off_bar = (uint32_t)o;
  o += (2 * dsa::kMaxStages + 2 * dsa::kMaxAccBufs + 2 * dsa::kMaxQBufs + 1) * 8;
  s->smem_bytes = o + 1024;  // slack for aligning the dynamic base to 1024
  return s->smem_bytes <= kSmemLimit;
}

template <int H>
int launch_score_h(const CUtensorMap& tk, const CUtensorMap& ts, const CUtensorMap& tq,
                   const dsa::ScoreParams& p, size_t smem, int grid, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(dsa::score_topk_kernel<H>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
  });
  if (attr_err != cudaSuccess)
    return fail(DSA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
  // programmatic stream serialisation: the kernel's prologue (TMEM
  // allocation, barrier set-up) overlaps the preceding plan or cache-write
  // kernel; it waits for that kernel's results before reading them
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(dsa::kScoreThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = env_int("DSA_PDL", 1, 0, 1);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, dsa::score_topk_kernel<H>, tk, ts, tq, p);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "score_topk_kernel launch: %s", cudaGetErrorString(e));
  return check_launch("score_topk_kernel");
}

int launch_score(int H, const CUtensorMap& tk, const CUtensorMap& ts, const CUtensorMap& tq,
                 const dsa::ScoreParams& p, size_t smem, int grid, cudaStream_t st) {
  switch (H) {
    case 4: return launch_score_h<4>(tk, ts, tq, p, smem, grid, st);
    case 8: return launch_score_h<8>(tk, ts, tq, p, smem, grid, st);
    case 16: return launch_score_h<16>(tk, ts, tq, p, smem, grid, st);
    case 32: return launch_score_h<32>(tk, ts, tq, p, smem, grid, st);
    case 64: return launch_score_h<64>(tk, ts, tq, p, smem, grid, st);
    case 128: return launch_score_h<128>(tk, ts, tq, p, smem, grid, st);
    default: return fail(DSA_ERR_UNSUPPORTED, "H=%d is not supported", H);
  }
}

// ---------------------------------------------------------------- shared pieces
struct Batch {
  int T, H, R, max_blocks, k, max_num_batched_tokens;
  int64_t num_pages;
  const int32_t *qsl, *seq_lens, *block_table;
  int32_t* topk;
  void* ws;
  size_t ws_bytes;
  int32_t* status;
  cudaStream_t st;
  int ratio = 1;  // tokens per cache entry (compressed indexer cache when > 1)
};

// Keys per workspace score row for a decode layout (G = 1) sized for
// contexts up to max_ctx: max_ctx rounded up to a multiple of 128 when that
// is at most kScoreRowMax (every row of such a batch then fits, so the plan
// always takes the row path and the row kernel is never launched for
// nothing); 0 otherwise, or when the rows would take more than 256 MB.
int score_stride_for(int T, int G, int64_t max_ctx) {
  if (G != 1 || max_ctx <= 0 || T <= 0 || max_ctx > dsa::kScoreRowMax) return 0;
  const int64_t s = (max_ctx + 127) / 128 * 128;
  if ((int64_t)T * s * 4 > (int64_t(256) << 20)) return 0;
  return (int)s;
}

// The score-row stride a caller's workspace holds: the largest stride whose
// layout fits in ws_bytes (the stride dsa_indexer_workspace_bytes sized it
// for, when the caller passed exactly that many bytes).
int score_stride_in(const Batch& b, int G, int n_cta) {
  if (G != 1 || b.T <= 0) return 0;
  const size_t base = dsa::ws_layout(b.T, b.R, G, b.k, n_cta, 0).total;
  if (b.ws_bytes <= base) return 0;
  int64_t s = (int64_t)((b.ws_bytes - base) / (4 * (size_t)b.T)) / 128 * 128;
  s = std::min<int64_t>(s, dsa::kScoreRowMax);
  while (s > 0 && dsa::ws_layout(b.T, b.R, G, b.k, n_cta, (int)s).total > b.ws_bytes) s -= 128;
  return s > 0 ? (int)s : 0;
}

int check_batch(const Batch& b) {
  if (b.T < 0) return fail(DSA_ERR_INVALID_ARG, "T=%d < 0", b.T);
  if (b.R < 1) return fail(DSA_ERR_INVALID_ARG, "R=%d < 1", b.R);
  if (b.ratio < 1) return fail(DSA_ERR_INVALID_ARG, "compress_ratio=%d < 1", b.ratio);
  if (!supported_heads(b.H)) return fail(DSA_ERR_UNSUPPORTED, "H=%d not in {4,8,16,32,64,128}", b.H);
  if (b.k < 1 || b.k > DSA_MAX_TOPK)
    return fail(DSA_ERR_UNSUPPORTED, "index_topk=%d outside [1, %d]", b.k, DSA_MAX_TOPK);
  if (b.T > b.max_num_batched_tokens)
    return fail(DSA_ERR_INVALID_ARG, "T=%d exceeds max_num_batched_tokens=%d", b.T,
                b.max_num_batched_tokens);
  if (b.max_blocks < 1) return fail(DSA_ERR_INVALID_ARG, "max_blocks=%d < 1", b.max_blocks);
  if (b.num_pages < 1 || b.num_pages > (int64_t)(INT32_MAX / (DSA_PAGE_BYTES / 128)))
    return fail(DSA_ERR_INVALID_ARG, "num_pages=%lld outside [1, %d]", (long long)b.num_pages,
                INT32_MAX / (DSA_PAGE_BYTES / 128));
  if (!b.qsl || !b.seq_lens || !b.block_table || !b.topk)
    return fail(DSA_ERR_INVALID_ARG, "null metadata or topk_buffer pointer");
  if (!b.ws) return fail(DSA_ERR_INVALID_ARG, "null workspace");
  if (!aligned(b.ws, 256)) return fail(DSA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t need = dsa_indexer_workspace_bytes(b.T, b.H, b.R, 0, b.k);
  if (b.ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", b.ws_bytes, need);
  return DSA_OK;
}

int launch_plan(const Batch& b, int G, int* launches) {
  dsa::PlanParams pp;
  pp.qsl = b.qsl;
  pp.seq_lens = b.seq_lens;
  pp.R = b.R;
  pp.T = b.T;
  pp.G = G;
  pp.max_blocks = b.max_blocks;
  pp.index_topk = b.k;
  pp.ratio = b.ratio;
  if (sm_count() <= 0) return fail(DSA_ERR_CUDA, "no CUDA device");
  pp.n_cta = grid_ctas();
  pp.min_tiles = env_int("DSA_MIN_SPLIT", 1024, 128, 1 << 20) / 128;
  pp.item_cost = env_int("DSA_ITEM_TILES", 2, 0, 64);
  pp.topk_buffer = b.topk;
  pp.ws = static_cast<unsigned char*>(b.ws);
  pp.L = dsa::ws_layout(b.T, b.R, G, b.k, pp.n_cta, score_stride_in(b, G, pp.n_cta));
  pp.status = b.status;
  dsa::plan_kernel<<<1, dsa::kPlanThreads, 0, b.st>>>(pp);
  ++*launches;
  return check_launch("plan_kernel");
}

struct LayerQ {
  const uint8_t* q_fp8;
  const float* q_scale;
  const float* w;
  const uint8_t* k_cache;
  float* scores_out;
  int64_t scores_ld;
};

// meta_ready: the launch right before this one is the layer's cache write, a
// plain launch issued after the plan, so the plan completed before it started:
// the scoring kernel may read the plan's outputs, and the cache entries below
// each request's first new entry, before its programmatic-launch wait.
// q_ready: that cache write does not produce q_fp8 (FP32-input layers).
int launch_score_layer(const Batch& b, const ScoreShape& s, const LayerQ& lq, int* launches,
                       bool meta_ready, bool q_ready) {
  // the pool as 128-byte rows: a page is rows [66 p, 66 p + 66), its 64 key
  // rows then 2 rows of scales; key boxes of 64 rows (swizzled into the MMA
  // operand layout), scale boxes of 2 rows (plain)
  CUtensorMap tk, ts, tq;
  int rc = make_rows128_map(&tk, lq.k_cache, (uint64_t)b.num_pages * (DSA_PAGE_BYTES / 128), 64);
  if (rc) return rc;
  rc = make_rows128_map(&ts, lq.k_cache, (uint64_t)b.num_pages * (DSA_PAGE_BYTES / 128), 2, false);
  if (rc) return rc;
  rc = make_rows128_map(&tq, lq.q_fp8, (uint64_t)b.T * b.H,
                        s.q_box_per_token ? (uint32_t)b.H : (uint32_t)(s.G * b.H));
  if (rc) return rc;
  const int grid = grid_ctas();
  const dsa::WsLayout L = dsa::ws_layout(b.T, b.R, s.G, b.k, grid, score_stride_in(b, s.G, grid));
  unsigned char* ws = static_cast<unsigned char*>(b.ws);
  dsa::ScoreParams p = s.offs;
  p.qsl = b.qsl;
  p.seq_lens = b.seq_lens;
  p.block_table = b.block_table;
  p.max_blocks = b.max_blocks;
  p.k_cache = lq.k_cache;
  p.num_pages = b.num_pages;
  p.q_scale = lq.q_scale;
  p.w = lq.w;
  p.T = b.T;
  p.H = b.H;
  p.G = s.G;
  p.k = b.k;
  p.C = s.C;
  p.NS = s.NS;
  p.NB = s.NB;
  p.NQ = s.NQ;
  p.NR = s.NR;
  p.BPS = s.BPS;
  p.lg_bps = s.lg_bps;
  p.lg_nb = s.lg_nb;
  p.lg_nr = s.lg_nr;
  p.ratio = b.ratio;
  p.q_bytes = s.q_bytes;
  p.n_max = s.n_max;
  p.q_box_per_token = s.q_box_per_token;
  p.meta_ready = meta_ready ? 1 : 0;
  p.q_ready = q_ready ? 1 : 0;
  p.items = reinterpret_cast<const dsa::Item*>(ws + L.items);
  p.cta_start = reinterpret_cast<const int32_t*>(ws + L.cta_start);
  p.heads = reinterpret_cast<const dsa::CtaHead*>(ws + L.heads);
  p.CB = L.cb;
  p.cand_keys = reinterpret_cast<uint32_t*>(ws + L.cand_keys);
  p.cand_idx = reinterpret_cast<int32_t*>(ws + L.cand_idx);
  p.cand_hist = reinterpret_cast<uint16_t*>(ws + L.cand_hist);
  p.cand_start = reinterpret_cast<uint16_t*>(ws + L.cand_start);
  p.ghist = reinterpret_cast<uint32_t*>(ws + L.ghist);
  p.wide_of = reinterpret_cast<const int32_t*>(ws + L.wide_of);
  p.cand_count = reinterpret_cast<int32_t*>(ws + L.cand_count);
  p.done = reinterpret_cast<int32_t*>(ws + L.done);
  p.topk = b.topk;
  p.scores_out = lq.scores_out;
  p.scores_ld = lq.scores_ld;
  p.score_rows = reinterpret_cast<uint32_t*>(ws + L.score_rows);
  p.score_stride = L.score_stride;
  p.status = b.status;
  p.wait_limit = (uint32_t)env_int("DSA_WAIT_LIMIT", (int)dsa::kWaitLimit, 0, (int)dsa::kWaitLimit);
  rc = launch_score(b.H, tk, ts, tq, p, s.smem_bytes, grid, b.st);
  if (rc == DSA_OK) ++*launches;
  return rc;
}

// The top-k of the rows the scoring kernel wrote into the workspace (decode
// layouts whose workspace has room for them; nothing to do otherwise).
int launch_rows_topk(const Batch& b, const ScoreShape& s, int* launches) {
  const int grid = grid_ctas();
  const dsa::WsLayout L = dsa::ws_layout(b.T, b.R, s.G, b.k, grid, score_stride_in(b, s.G, grid));
  if (L.score_stride <= 0) return DSA_OK;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(dsa::rows_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)dsa::rows_topk_smem(dsa::kScoreRowMax));
  });
  if (attr_err != cudaSuccess)
    return fail(DSA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
  unsigned char* ws = static_cast<unsigned char*>(b.ws);
  dsa::RowsTopkParams rp;
  rp.score_rows = reinterpret_cast<const uint32_t*>(ws + L.score_rows);
  rp.row_keys = reinterpret_cast<const int32_t*>(ws + L.row_keys);
  rp.score_stride = L.score_stride;
  rp.k = b.k;
  rp.topk = b.topk;
  // programmatic stream serialisation: the row kernel's blocks are placed
  // while the scoring kernel drains; they wait for its keys before reading
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)b.T);
  cfg.blockDim = dim3(dsa::kRowsThreads);
  cfg.dynamicSmemBytes = dsa::rows_topk_smem(L.score_stride);
  cfg.stream = b.st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = env_int("DSA_PDL", 1, 0, 1);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, dsa::rows_topk_kernel, rp);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "rows_topk_kernel launch: %s", cudaGetErrorString(e));
  ++*launches;
  return check_launch("rows_topk_kernel");
}

// Record a caller's timing event on the stream; inside stream capture it must
// become an event-record node of the graph (external event), otherwise the
// event would only express a dependency and never be recorded on replay.
cudaError_t record_event(void* ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags((cudaEvent_t)ev, st, cudaEventRecordExternal);
  return cudaEventRecord((cudaEvent_t)ev, st);
}

// Cache write of T new keys (FP32 or BF16); with q given (BF16 only) the same
// launch also quantises the T*H query blocks into q_fp8 / q_scale.
template <typename TIn>
int launch_write_t(const TIn* k, const Batch& b, uint8_t* k_cache, int64_t* slot_mapping,
                   const TIn* q, int H, uint8_t* q_fp8, float* q_scale, int* launches) {
  const int warps_per_block = 8;
  const int64_t warps = (int64_t)b.T + (q ? (int64_t)b.T * H : 0);
  const int64_t grid = (warps + warps_per_block - 1) / warps_per_block;
  if (grid > INT32_MAX) return fail(DSA_ERR_INVALID_ARG, "too many rows for one cache-write launch");
  // a plain launch (no programmatic serialisation): a layer stack's scoring
  // launch relies on it to read the plan's outputs before its own wait
  dsa::write_k_kernel<TIn><<<(unsigned)grid, 32 * warps_per_block, 0, b.st>>>(
      k, b.T, b.qsl, b.seq_lens, b.R, b.block_table, b.max_blocks, k_cache, b.num_pages,
      b.ratio, slot_mapping, b.status, q, H, q_fp8, q_scale);
  ++*launches;
  return check_launch("write_k_kernel");
}

int launch_write(const float* k, const Batch& b, uint8_t* k_cache, int64_t* slot_mapping,
                 int* launches) {
  return launch_write_t<float>(k, b, k_cache, slot_mapping, nullptr, 0, nullptr, nullptr,
                               launches);
}

__global__ void copy_rows_kernel(const int4* __restrict__ src, int4* __restrict__ dst, int64_t n16) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// ---------------------------------------------------------------- built-in workspace
// Workspace for callers that cannot allocate device memory.  It is a
// file-scope device array, so every GPU that loads this library holds it
// until the process exits.  Host code must not use the symbol itself as a
// device address (on the host it is only a stand-in): the real address is
// looked up with cudaGetSymbolAddress while the device is current, on the
// first call on that device, and cached together with the identity of the
// device's current context, so that a call after a device reset (a new
// context, in which the array may sit elsewhere) looks it up again.
constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_ws_mutex;
void* g_static_ws_ptr[kMaxDevices] = {};
unsigned long long g_static_ws_ctx[kMaxDevices] = {};

// Unique id of the calling thread's current context (0 if unavailable).
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DSA_ERR_UNSUPPORTED, "device %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_static_ws_mutex);
  // the runtime makes the device's primary context current on first use
  if (!g_static_ws_ptr[dev]) {
    e = cudaFree(nullptr);
    if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "device %d: %s", dev, cudaGetErrorString(e));
  }
  const unsigned long long ctx = current_context_id();
  if (!g_static_ws_ptr[dev] || g_static_ws_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || !p)
      return fail(DSA_ERR_CUDA, "cudaGetSymbolAddress of the built-in workspace: %s",
                  cudaGetErrorString(e));
    g_static_ws_ptr[dev] = p;
    g_static_ws_ctx[dev] = ctx;
  }
  *out = g_static_ws_ptr[dev];
  return DSA_OK;
}

// ---------------------------------------------------------------- layer stacks
// The two layer-input forms (FP32 keys + quantised queries, or BF16 keys and
// queries quantised by the cache-write launch) share one stack driver.
int check_layer(const dsa_layer_io& io, int l) {
  if (!io.k || !io.q_fp8 || !io.q_scale || !io.w || !io.k_cache)
    return fail(DSA_ERR_INVALID_ARG, "F layer %d has a null input", l);
  if (!aligned(io.k, 16) || !aligned(io.q_fp8, 16) || !aligned(io.k_cache, 16))
    return fail(DSA_ERR_INVALID_ARG, "F layer %d: k, q_fp8, k_cache must be 16-byte aligned", l);
  return DSA_OK;
}
int check_layer(const dsa_layer_io_bf16& io, int l) {
  if (!io.k || !io.q || !io.w || !io.k_cache || !io.q_fp8 || !io.q_scale)
    return fail(DSA_ERR_INVALID_ARG, "F layer %d has a null input", l);
  if (!aligned(io.k, 16) || !aligned(io.q, 16) || !aligned(io.q_fp8, 16) || !aligned(io.k_cache, 16))
    return fail(DSA_ERR_INVALID_ARG, "F layer %d: k, q, q_fp8, k_cache must be 16-byte aligned", l);
  return DSA_OK;
}
int write_layer(const dsa_layer_io& io, const Batch& b, int64_t* slot_mapping, int* launches) {
  return launch_write(io.k, b, io.k_cache, slot_mapping, launches);
}
int write_layer(const dsa_layer_io_bf16& io, const Batch& b, int64_t* slot_mapping, int* launches) {
  return launch_write_t<uint16_t>(static_cast<const uint16_t*>(io.k), b, io.k_cache, slot_mapping,
                                  static_cast<const uint16_t*>(io.q), b.H, io.q_fp8, io.q_scale,
                                  launches);
}

// FP32-input layers take q_fp8 as an input; BF16-input layers have the cache
// write quantise it.
template <typename IO> struct QueriesAreInputs;
template <> struct QueriesAreInputs<dsa_layer_io> { static constexpr bool value = true; };
template <> struct QueriesAreInputs<dsa_layer_io_bf16> { static constexpr bool value = false; };

template <typename IO>
int stack_run(int num_layers, const char* pattern, int freq, int offset, const IO* layers,
              const Batch& b, int32_t* const* per_layer_topk_out, int64_t* slot_mapping) {
  g_last_launches = 0;
  if (num_layers < 1) return fail(DSA_ERR_INVALID_ARG, "num_layers=%d < 1", num_layers);
  if (!layers) return fail(DSA_ERR_INVALID_ARG, "null layers array");
  int rc = check_batch(b);
  if (rc) return rc;
  // schedule and per-layer inputs are checked before anything is launched
  for (int l = 0; l < num_layers; ++l) {
    const int full = dsa_layer_is_full(l, pattern, freq, offset);
    if (full < 0) return full;
    if (l == 0 && !full)
      return fail(DSA_ERR_INVALID_ARG,
                  "layer 0 is S: no F layer has written the top-k buffer in this pass");
    if (full && (rc = check_layer(layers[l], l)) != DSA_OK) return rc;
  }
  if (b.T == 0) return DSA_OK;
  ScoreShape s;
  if (!score_shape(b.T, b.R, b.H, b.k, &s))
    return fail(DSA_ERR_UNSUPPORTED, "no shared-memory configuration for H=%d, index_topk=%d", b.H,
                b.k);
  int launches = 0;
  rc = launch_plan(b, s.G, &launches);
  bool first_full = true;
  for (int l = 0; l < num_layers && rc == DSA_OK; ++l) {
    const int full = dsa_layer_is_full(l, pattern, freq, offset);
    if (full) {
      const IO& io = layers[l];
      rc = write_layer(io, b, first_full ? slot_mapping : nullptr, &launches);
      first_full = false;
      if (rc) break;
      LayerQ lq{io.q_fp8, io.q_scale, io.w, io.k_cache, nullptr, 0};
      if (io.score_begin && record_event(io.score_begin, b.st) != cudaSuccess) {
        rc = fail(DSA_ERR_CUDA, "recording score_begin of layer %d failed", l);
        break;
      }
      // the cache write, a plain launch, lies between the plan and this launch
      rc = launch_score_layer(b, s, lq, &launches, true, QueriesAreInputs<IO>::value);
      if (rc) break;
      rc = launch_rows_topk(b, s, &launches);
      if (rc) break;
      if (io.score_end && record_event(io.score_end, b.st) != cudaSuccess) {
        rc = fail(DSA_ERR_CUDA, "recording score_end of layer %d failed", l);
        break;
      }
    }
    if (per_layer_topk_out && per_layer_topk_out[l]) {
      const int64_t bytes = (int64_t)b.T * b.k * 4;
      if (bytes % 16 == 0 && aligned(per_layer_topk_out[l], 16) && aligned(b.topk, 16)) {
        copy_rows_kernel<<<256, 256, 0, b.st>>>(reinterpret_cast<const int4*>(b.topk),
                                                reinterpret_cast<int4*>(per_layer_topk_out[l]),
                                                bytes / 16);
        ++launches;
        rc = check_launch("copy_rows_kernel");
      } else {
        if (cudaMemcpyAsync(per_layer_topk_out[l], b.topk, (size_t)bytes,
                            cudaMemcpyDeviceToDevice, b.st) != cudaSuccess)
          rc = fail(DSA_ERR_CUDA, "snapshot copy of layer %d failed", l);
      }
    }
  }
  g_last_launches = launches;
  return rc;
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

int dsa_abi_version(void) { return 100; }

const char* dsa_last_error(void) { return g_last_error.c_str(); }

int dsa_last_launch_count(void) { return g_last_launches; }

int dsa_layer_is_full(int layer_id, const char* pattern, int freq, int offset) {
  if (layer_id < 0) return fail(DSA_ERR_INVALID_ARG, "layer_id=%d < 0", layer_id);
  if (pattern) {
    const size_t n = strlen(pattern);
    for (size_t i = 0; i < n; ++i)
      if (pattern[i] != 'F' && pattern[i] != 'S')
        return fail(DSA_ERR_INVALID_ARG, "pattern character %zu is '%c', not F or S", i,
                    pattern[i]);
    if ((size_t)layer_id >= n) return 1;  // beyond the pattern: F
    return pattern[layer_id] == 'F' ? 1 : 0;
  }
  if (freq <= 0) return fail(DSA_ERR_INVALID_ARG, "index_topk_freq=%d <= 0", freq);
  int x = layer_id - offset + 1;
  if (x < 0) x = 0;
  return (x % freq) == 0 ? 1 : 0;
}

size_t dsa_indexer_workspace_bytes(int T, int H, int R, int64_t max_ctx, int index_topk) {
  if (T < 0 || R < 1 || !supported_heads(H) || index_topk < 1 || index_topk > DSA_MAX_TOPK)
    return 0;
  const int G = choose_group(T, R, H, index_topk);
  return dsa::ws_layout(T, R, G, index_topk, grid_ctas(), score_stride_for(T, G, max_ctx)).total;
}

int dsa_quantize_fp8_blocks(const float* x, int64_t n_blocks, uint8_t* codes, float* scales,
                            dsa_stream_t stream) {
  g_last_launches = 0;
  if (n_blocks < 0) return fail(DSA_ERR_INVALID_ARG, "n_blocks < 0");
  if (n_blocks == 0) return DSA_OK;
  if (!x || !codes || !scales) return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(x, 16) || !aligned(codes, 4))
    return fail(DSA_ERR_INVALID_ARG, "x must be 16-byte and codes 4-byte aligned");
  const int64_t threads = n_blocks * 32;
  const int64_t grid = (threads + 255) / 256;
  if (grid > INT32_MAX) return fail(DSA_ERR_INVALID_ARG, "too many blocks");
  dsa::quantize_blocks_kernel<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(x, n_blocks, codes,
                                                                                scales);
  g_last_launches = 1;
  return check_launch("quantize_blocks_kernel");
}

int dsa_indexer_write_k(const float* k, int T, const int32_t* query_start_loc,
                        const int32_t* seq_lens, int R, const int32_t* block_table,
                        int max_blocks, uint8_t* k_cache, int64_t num_pages,
                        int64_t* slot_mapping, int32_t* dev_status, dsa_stream_t stream) {
  return dsa_indexer_write_k_compressed(k, T, query_start_loc, seq_lens, R, block_table,
                                        max_blocks, k_cache, num_pages, 1, slot_mapping,
                                        dev_status, stream);
}

int dsa_indexer_write_k_compressed(const float* k, int T, const int32_t* query_start_loc,
                                   const int32_t* seq_lens, int R, const int32_t* block_table,
                                   int max_blocks, uint8_t* k_cache, int64_t num_pages,
                                   int compress_ratio, int64_t* slot_mapping,
                                   int32_t* dev_status, dsa_stream_t stream) {
  g_last_launches = 0;
  if (compress_ratio < 1) return fail(DSA_ERR_INVALID_ARG, "compress_ratio=%d < 1", compress_ratio);
  if (T < 0) return fail(DSA_ERR_INVALID_ARG, "T=%d < 0", T);
  if (R < 1) return fail(DSA_ERR_INVALID_ARG, "R=%d < 1", R);
  if (max_blocks < 1) return fail(DSA_ERR_INVALID_ARG, "max_blocks < 1");
  if (num_pages < 1) return fail(DSA_ERR_INVALID_ARG, "num_pages < 1");
  if (T == 0) return DSA_OK;
  if (!k || !query_start_loc || !seq_lens || !block_table || !k_cache)
    return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k, 16) || !aligned(k_cache, 16))
    return fail(DSA_ERR_INVALID_ARG, "k and k_cache must be 16-byte aligned");
  Batch b{};
  b.T = T;
  b.R = R;
  b.max_blocks = max_blocks;
  b.num_pages = num_pages;
  b.qsl = query_start_loc;
  b.seq_lens = seq_lens;
  b.block_table = block_table;
  b.status = dev_status;
  b.st = (cudaStream_t)stream;
  b.ratio = compress_ratio;
  int launches = 0;
  const int rc = launch_write(k, b, k_cache, slot_mapping, &launches);
  g_last_launches = launches;
  return rc;
}

int dsa_indexer_score_topk(const uint8_t* q_fp8, const float* q_scale, const float* w, int T,
                           int H, const uint8_t* k_cache, int64_t num_pages,
                           const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                           const int32_t* block_table, int max_blocks, int index_topk,
                           int32_t* topk_buffer, int max_num_batched_tokens, float* scores_out,
                           int64_t scores_ld, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, dsa_stream_t stream) {
  return dsa_indexer_score_topk_compressed(q_fp8, q_scale, w, T, H, k_cache, num_pages,
                                           query_start_loc, seq_lens, R, block_table, max_blocks,
                                           1, index_topk, topk_buffer, max_num_batched_tokens,
                                           scores_out, scores_ld, workspace, workspace_bytes,
                                           dev_status, stream);
}

int dsa_indexer_score_topk_compressed(const uint8_t* q_fp8, const float* q_scale, const float* w,
                                      int T, int H, const uint8_t* k_cache, int64_t num_pages,
                                      const int32_t* query_start_loc, const int32_t* seq_lens,
                                      int R, const int32_t* block_table, int max_blocks,
                                      int compress_ratio, int index_topk, int32_t* topk_buffer,
                                      int max_num_batched_tokens, float* scores_out,
                                      int64_t scores_ld, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_status, dsa_stream_t stream) {
  g_last_launches = 0;
  Batch b{T, H, R, max_blocks, index_topk, max_num_batched_tokens, num_pages, query_start_loc,
          seq_lens, block_table, topk_buffer, workspace, workspace_bytes, dev_status,
          (cudaStream_t)stream, compress_ratio};
  int rc = check_batch(b);
  if (rc) return rc;
  if (T == 0) return DSA_OK;
  if (!q_fp8 || !q_scale || !w || !k_cache) return fail(DSA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(q_fp8, 16) || !aligned(k_cache, 16))
    return fail(DSA_ERR_INVALID_ARG, "q_fp8 and k_cache must be 16-byte aligned");
  if (scores_out && scores_ld < 1) return fail(DSA_ERR_INVALID_ARG, "scores_ld < 1");
  ScoreShape s;
  if (!score_shape(T, R, H, index_topk, &s))
    return fail(DSA_ERR_UNSUPPORTED, "no shared-memory configuration for H=%d, index_topk=%d", H,
                index_topk);
  int launches = 0;
  rc = launch_plan(b, s.G, &launches);
  if (rc == DSA_OK) {
    LayerQ lq{q_fp8, q_scale, w, k_cache, scores_out, scores_ld};
    rc = launch_score_layer(b, s, lq, &launches, false, true);
    if (rc == DSA_OK) rc = launch_rows_topk(b, s, &launches);
  }
  g_last_launches = launches;
  return rc;
}

int dsa_indexer_score_topk_no_alloc(const uint8_t* q_fp8, const float* q_scale, const float* w,
                                    int T, int H, const uint8_t* k_cache, int64_t num_pages,
                                    const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                                    const int32_t* block_table, int max_blocks, int index_topk,
                                    int32_t* topk_buffer, int max_num_batched_tokens,
                                    int32_t* dev_status, dsa_stream_t stream) {
  g_last_launches = 0;
  // the same argument checks, in the same order, as dsa_indexer_score_topk
  // (a stand-in workspace of the built-in size: its address is not used)
  Batch b{T, H, R, max_blocks, index_topk, max_num_batched_tokens, num_pages, query_start_loc,
          seq_lens, block_table, topk_buffer, reinterpret_cast<void*>(uintptr_t(256)),
          ~size_t(0), dev_status, (cudaStream_t)stream, 1};
  int rc = check_batch(b);
  if (rc) return rc;
  const size_t need = dsa_indexer_workspace_bytes(T, H, R, 0, index_topk);
  if (need > kStaticWorkspaceBytes)
    return fail(DSA_ERR_WORKSPACE_TOO_SMALL,
                "this batch needs %zu bytes of workspace; the built-in workspace holds %zu "
                "(use dsa_indexer_score_topk with a caller-provided workspace)",
                need, kStaticWorkspaceBytes);
  void* ws = nullptr;
  rc = static_workspace(&ws);
  if (rc) return rc;
  return dsa_indexer_score_topk(q_fp8, q_scale, w, T, H, k_cache, num_pages, query_start_loc,
                                seq_lens, R, block_table, max_blocks, index_topk, topk_buffer,
                                max_num_batched_tokens, nullptr, 0, ws, kStaticWorkspaceBytes,
                                dev_status, stream);
}

size_t dsa_indexer_no_alloc_workspace_bytes(void) { return kStaticWorkspaceBytes; }

int dsa_layer_stack_run(int num_layers, const char* pattern, int freq, int offset,
                        const dsa_layer_io* layers, int T, int H,
                        const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                        const int32_t* block_table, int max_blocks, int64_t num_pages,
                        int index_topk, int32_t* topk_buffer, int max_num_batched_tokens,
                        int32_t* const* per_layer_topk_out, int64_t* slot_mapping,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        dsa_stream_t stream) {
  const Batch b{T, H, R, max_blocks, index_topk, max_num_batched_tokens, num_pages,
                query_start_loc, seq_lens, block_table, topk_buffer, workspace, workspace_bytes,
                dev_status, (cudaStream_t)stream};
  return stack_run(num_layers, pattern, freq, offset, layers, b, per_layer_topk_out, slot_mapping);
}

int dsa_layer_stack_run_compressed(int num_layers, const char* pattern, int freq, int offset,
                                   const dsa_layer_io* layers, int T, int H,
                                   const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                                   const int32_t* block_table, int max_blocks, int64_t num_pages,
                                   int compress_ratio, int index_topk, int32_t* topk_buffer,
                                   int max_num_batched_tokens, int32_t* const* per_layer_topk_out,
                                   int64_t* slot_mapping, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, dsa_stream_t stream) {
  const Batch b{T, H, R, max_blocks, index_topk, max_num_batched_tokens, num_pages,
                query_start_loc, seq_lens, block_table, topk_buffer, workspace, workspace_bytes,
                dev_status, (cudaStream_t)stream, compress_ratio};
  return stack_run(num_layers, pattern, freq, offset, layers, b, per_layer_topk_out, slot_mapping);
}

int dsa_layer_stack_run_bf16(int num_layers, const char* pattern, int freq, int offset,
                             const dsa_layer_io_bf16* layers, int T, int H,
                             const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                             const int32_t* block_table, int max_blocks, int64_t num_pages,
                             int index_topk, int32_t* topk_buffer, int max_num_batched_tokens,
                             int32_t* const* per_layer_topk_out, int64_t* slot_mapping,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             dsa_stream_t stream) {
  const Batch b{T, H, R, max_blocks, index_topk, max_num_batched_tokens, num_pages,
                query_start_loc, seq_lens, block_table, topk_buffer, workspace, workspace_bytes,
                dev_status, (cudaStream_t)stream};
  return stack_run(num_layers, pattern, freq, offset, layers, b, per_layer_topk_out, slot_mapping);
}

int dsa_indexer_write_k_bf16(const void* k, int T, const int32_t* query_start_loc,
                             const int32_t* seq_lens, int R, const int32_t* block_table,
                             int max_blocks, uint8_t* k_cache, int64_t num_pages,
                             const void* q, int H, uint8_t* q_fp8, float* q_scale,
                             int64_t* slot_mapping, int32_t* dev_status, dsa_stream_t stream) {
  g_last_launches = 0;
  if (T < 0) return fail(DSA_ERR_INVALID_ARG, "T=%d < 0", T);
  if (R < 1) return fail(DSA_ERR_INVALID_ARG, "R=%d < 1", R);
  if (max_blocks < 1) return fail(DSA_ERR_INVALID_ARG, "max_blocks < 1");
  if (num_pages < 1) return fail(DSA_ERR_INVALID_ARG, "num_pages < 1");
  if (q && (H < 1 || !q_fp8 || !q_scale))
    return fail(DSA_ERR_INVALID_ARG, "with q: H >= 1 and q_fp8, q_scale outputs are required");
  if (T == 0) return DSA_OK;
  if (!k || !query_start_loc || !seq_lens || !block_table || !k_cache)
    return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(k, 16) || !aligned(k_cache, 16) || (q && (!aligned(q, 16) || !aligned(q_fp8, 16))))
    return fail(DSA_ERR_INVALID_ARG, "k, q, q_fp8 and k_cache must be 16-byte aligned");
  Batch b{};
  b.T = T;
  b.H = H;
  b.R = R;
  b.max_blocks = max_blocks;
  b.num_pages = num_pages;
  b.qsl = query_start_loc;
  b.seq_lens = seq_lens;
  b.block_table = block_table;
  b.status = dev_status;
  b.st = (cudaStream_t)stream;
  int launches = 0;
  const int rc = launch_write_t<uint16_t>(static_cast<const uint16_t*>(k), b, k_cache, slot_mapping,
                                          static_cast<const uint16_t*>(q), H, q_fp8, q_scale,
                                          &launches);
  g_last_launches = launches;
  return rc;
}

int dsa_mla_write_kv(const float* kv, int T, const int32_t* query_start_loc,
                     const int32_t* seq_lens, int R, const int32_t* block_table, int max_blocks,
                     uint8_t* kv_cache, int64_t num_pages, int64_t* slot_mapping,
                     int32_t* dev_status, dsa_stream_t stream) {
  g_last_launches = 0;
  if (T < 0) return fail(DSA_ERR_INVALID_ARG, "T=%d < 0", T);
  if (R < 1) return fail(DSA_ERR_INVALID_ARG, "R=%d < 1", R);
  if (max_blocks < 1) return fail(DSA_ERR_INVALID_ARG, "max_blocks < 1");
  if (num_pages < 1) return fail(DSA_ERR_INVALID_ARG, "num_pages < 1");
  if (T == 0) return DSA_OK;
  if (!kv || !query_start_loc || !seq_lens || !block_table || !kv_cache)
    return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(kv, 16) || !aligned(kv_cache, 16))
    return fail(DSA_ERR_INVALID_ARG, "kv and kv_cache must be 16-byte aligned");
  const int64_t grid = ((int64_t)T * 32 + 255) / 256;
  if (grid > INT32_MAX) return fail(DSA_ERR_INVALID_ARG, "too many rows");
  dsa::mla_write_kernel<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(
      kv, T, query_start_loc, seq_lens, R, block_table, max_blocks, kv_cache, num_pages,
      slot_mapping, dev_status);
  g_last_launches = 1;
  return check_launch("mla_write_kernel");
}

int dsa_sparse_mla_attention(const void* q, int T, int Hq, const uint8_t* kv_cache,
                             int64_t num_pages, const int32_t* query_start_loc,
                             const int32_t* seq_lens, int R, const int32_t* block_table,
                             int max_blocks, const int32_t* topk_indices, int index_topk,
                             float softmax_scale, void* out, float* lse, int32_t* dev_status,
                             dsa_stream_t stream) {
  g_last_launches = 0;
  if (T < 0) return fail(DSA_ERR_INVALID_ARG, "T=%d < 0", T);
  if (R < 1) return fail(DSA_ERR_INVALID_ARG, "R=%d < 1", R);
  if (Hq < 1 || Hq > dsa::kMlaMaxHeads)
    return fail(DSA_ERR_UNSUPPORTED, "Hq=%d outside [1, %d]", Hq, dsa::kMlaMaxHeads);
  if (index_topk < 1 || index_topk > dsa::kMlaMaxTopk)
    return fail(DSA_ERR_UNSUPPORTED, "index_topk=%d outside [1, %d]", index_topk,
                dsa::kMlaMaxTopk);
  if (max_blocks < 1) return fail(DSA_ERR_INVALID_ARG, "max_blocks < 1");
  if (num_pages < 1 || num_pages > INT32_MAX / DSA_PAGE_TOKENS)
    return fail(DSA_ERR_INVALID_ARG, "num_pages=%lld outside [1, %d]", (long long)num_pages,
                INT32_MAX / DSA_PAGE_TOKENS);
  if (!(softmax_scale > 0.0f) || !(softmax_scale < 1e30f))
    return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
  if (T == 0) return DSA_OK;
  if (!q || !kv_cache || !query_start_loc || !seq_lens || !block_table || !topk_indices || !out)
    return fail(DSA_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16))
    return fail(DSA_ERR_INVALID_ARG, "q, kv_cache and out must be 16-byte aligned");
  if ((int64_t)T * 4 > INT32_MAX) return fail(DSA_ERR_INVALID_ARG, "too many rows");
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(dsa::sparse_mla_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)dsa::kMlaSmemBytes);
  });
  if (attr_err != cudaSuccess)
    return fail(DSA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
  dsa::MlaParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.cache = kv_cache;
  p.num_pages = num_pages;
  p.qsl = query_start_loc;
  p.seq_lens = seq_lens;
  p.R = R;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.topk = topk_indices;
  p.k = index_topk;
  p.T = T;
  p.Hq = Hq;
  p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.status = dev_status;
  // four CTAs per row, one per 128-wide quarter of the output
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(T * dsa::kMlaQuarters));
  cfg.blockDim = dim3(dsa::kMlaThreads);
  cfg.dynamicSmemBytes = dsa::kMlaSmemBytes;
  cfg.stream = (cudaStream_t)stream;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, dsa::sparse_mla_kernel, p);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "sparse_mla_kernel launch: %s", cudaGetErrorString(e));
  g_last_launches = 1;
  return check_launch("sparse_mla_kernel");
}

}  // extern "C"
