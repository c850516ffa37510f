// Sparse MLA attention over the indexer's top-k rows, and the cache write of
// its 656-byte fp8_ds_mla records.
//
// Record ("GLM-5.3 推理全链路(十二)", the list above the byte-accounting table):
// a token's 512-d KV latent and 64-d RoPE part as 576 E4M3 bytes, then 16 B of
// FP32 scales for each of five 128-element blocks -- one scale per 32
// elements, 20 slots of which the last two (the half-filled RoPE block) are
// padding, written as 0.  64 records back to back form a 41,984-byte page,
// addressed through the indexer's block table (the two caches share slot
// numbers).
//
// Attention ("RFC: DeepseekV32 模型适配支持" §2.1.3: the top-k is a 0 / -inf mask
// on the q.k scores, i.e. attention over the selected tokens only), absorbed
// MLA form: for query row t and head h, out[t,h] = sum_s softmax_s(scale *
// q[t,h] . key_s) * key_s[0:512] over the tokens s of row t of the top-k
// buffer (entries >= 0), lse[t,h] = ln sum_s exp(scale * q[t,h] . key_s).
//
// One CTA per (query row, 128-wide quarter of the 512 output dimensions): the
// FP32 output of 128 heads x 512 dimensions alone would fill all 512 columns
// of tensor memory, so each CTA keeps a quarter of it (128 columns), next to
// the row's queries (288 columns: the MMA's A operand, held in tensor memory
// so that it is not re-read from shared memory for every key tile), one
// 64-token score tile (64) and its BF16 probabilities (32).  The four CTAs
// of a row compute the same scores.  A tcgen05.mma costs its issuing thread
// ~45 cycles however small N is, and an M128 x N64 x K16 BF16 product takes
// the tensor core about as long, so key tiles are 64 tokens wide (the widest
// that fits next to the output quarter) and the 36 QK^T instructions of a
// tile are issued back to back from precomputed descriptors.
//   warps 0-3   softmax: thread = head; online softmax over 64-token tiles
//               (rescaling the output only when the running maximum grows by
//               more than 2^8), probabilities to tensor memory as BF16,
//               final normalisation and the BF16 output rows;
//   warps 4-9   converters: compact the top-k row and resolve its slots;
//               then dequantise each 32-token half tile of records to BF16
//               in shared memory (128-byte-swizzled rows, the K-major layout
//               of the QK^T B operand and the MN-major layout of the PV B
//               operand at once);
//   warp 10     MMA issuer: S = Q K^T (M = 128 heads, N = 64 tokens, K = 576)
//               and O += P V (N = 128 dimensions, K = 64 tokens);
//   warp 11     loader: the selected records into a ring of raw half tiles.
//
// Each CTA gathers the records of its row's half tiles into its own shared
// memory with one bulk copy per record (the four CTAs of a row read the same
// records; three of the four reads hit L2), and a raw slot is refilled once
// its own converters have dequantised it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "kwrite.cuh"

namespace dsa {

constexpr int kMlaDim = 576;
constexpr int kMlaLatent = 512;
constexpr int kMlaGroup = 32;
constexpr int kMlaScaleSlots = 20;
constexpr int kMlaRecBytes = 656;
constexpr int kMlaPageBytes = kPageTokens * kMlaRecBytes;  // 41,984
constexpr int kMlaMaxHeads = 128;
constexpr int kMlaMaxTopk = 2048;

// ---------------------------------------------------------------- cache write
// One warp per new token: lane l owns the float4s l, l+32, ..., l+128 of the
// 576-vector; the 8 lanes that share a 32-element group reduce its maximum.
__global__ void __launch_bounds__(256) mla_write_kernel(
    const float* __restrict__ kv, int T, const int32_t* __restrict__ qsl,
    const int32_t* __restrict__ seq_lens, int R, const int32_t* __restrict__ block_table,
    int max_blocks, uint8_t* __restrict__ cache, int64_t num_pages,
    int64_t* __restrict__ slot_mapping, int32_t* status) {
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const int t = (int)warp;
  const int r = find_request(qsl, R, t);
  const int q_begin = __ldg(qsl + r);
  const int q_len = __ldg(qsl + r + 1) - q_begin;
  const int seq_len = __ldg(seq_lens + r);
  const int pos = seq_len - q_len + (t - q_begin);
  int64_t slot = -1;
  if (q_len < 0 || seq_len < q_len || pos < 0 || pos >= seq_len || pos / kPageTokens >= max_blocks) {
    if (lane == 0) raise_status(status, kStatusBadMetadata);
  } else {
    const int64_t page = __ldg(block_table + (int64_t)r * max_blocks + pos / kPageTokens);
    if (page < 0 || page >= num_pages) {
      if (lane == 0) raise_status(status, kStatusBadPage);
    } else {
      uint8_t* rec = cache + page * kMlaPageBytes + (int64_t)(pos % kPageTokens) * kMlaRecBytes;
      const float4* src = reinterpret_cast<const float4*>(kv + (int64_t)t * kMlaDim);
#pragma unroll
      for (int i = 0; i < 5; ++i) {
        const int f = lane + 32 * i;           // float4 index; group f / 8
        const bool have = f < kMlaDim / 4;     // the last round covers 16 float4s
        const float4 v = have ? __ldg(src + f) : make_float4(0.f, 0.f, 0.f, 0.f);
        float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
        const uint32_t c01 = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(v.x, s), __fdiv_rn(v.y, s)), __NV_SATFINITE, __NV_E4M3);
        const uint32_t c23 = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(v.z, s), __fdiv_rn(v.w, s)), __NV_SATFINITE, __NV_E4M3);
        if (have) {
          reinterpret_cast<uint32_t*>(rec)[f] = (c01 & 0xFFFFu) | ((c23 & 0xFFFFu) << 16);
          if ((f & 7) == 0) reinterpret_cast<float*>(rec + kMlaDim)[f / 8] = s;
        }
      }
      if (lane < 2) reinterpret_cast<float*>(rec + kMlaDim)[18 + lane] = 0.0f;
      slot = page * kPageTokens + pos % kPageTokens;
    }
  }
  if (slot_mapping && lane == 0) slot_mapping[t] = slot;
}

// ---------------------------------------------------------------- attention
constexpr int kMlaTile = 64;                       // tokens per key tile (N of QK^T)
constexpr int kMlaHalf = 32;                       // tokens per raw half tile
constexpr int kMlaStages = 2;
constexpr int kMlaChunkBytes = kMlaTile * 128;     // 64 dimensions x 64 tokens, BF16
constexpr int kMlaStageBytes = 9 * kMlaChunkBytes; // 73,728
constexpr int kMlaRawStages = 3;
constexpr int kMlaRawBytes = kMlaHalf * kMlaRecBytes;  // 20,992: 32 records
constexpr int kMlaSoftmaxWarps = 4, kMlaProducerWarps = 6;  // 12 warps: 170 registers each
constexpr int kMlaThreads = (kMlaSoftmaxWarps + kMlaProducerWarps + 2) * 32;
constexpr int kMlaProducers = kMlaProducerWarps * 32;
constexpr int kMlaMmaWarp = kMlaSoftmaxWarps + kMlaProducerWarps;
constexpr int kMlaLoaderWarp = kMlaMmaWarp + 1;
constexpr int kMlaQuarters = 4;                      // CTAs per query row (128 output dimensions each)
// tensor-memory columns
constexpr uint32_t kMlaColO = 0;       // 128 FP32: this CTA's quarter of the output
constexpr uint32_t kMlaColS = 128;     // 64 FP32: the score tile
constexpr uint32_t kMlaColP = 192;     // 32: the tile's BF16 probabilities (A of PV)
constexpr uint32_t kMlaColQ = 224;     // 288: BF16 queries (A of QK^T)
constexpr float kMlaRescaleLog2 = 8.0f;  // rescale the output when the max grows by > 2^8

struct MlaParams {
  const uint16_t* q;            // [T, Hq, 576] BF16
  const uint8_t* cache;         // [num_pages, 41984]
  int64_t num_pages;
  const int32_t* qsl;
  const int32_t* seq_lens;
  int R;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* topk;          // [>= T, k]
  int k;
  int T, Hq;
  float scale_log2;             // softmax_scale * log2(e)
  uint16_t* out;                // [T, Hq, 512] BF16
  float* lse;                   // [T, Hq] or null
  int32_t* status;
};

struct MlaSmem {
  int32_t slot[kMlaMaxTopk];    // the row's selected tokens, compacted: page * 64 + offset, or -1
  int32_t warp_count[kMlaProducerWarps];
  int32_t n_valid;
  int32_t abort;
  int32_t conv_fail;            // set by a converter whose wait gave up; read after a barrier
  uint32_t tmem_base;
  uint32_t raw_live[kMlaRawStages];  // per raw half tile: bit n = record n is being copied
  uint64_t kfull[kMlaStages], kempty[kMlaStages];
  uint64_t rfull[kMlaRawStages], rempty[kMlaRawStages];
  uint64_t sfull, sfree, pfull, pvdone;
  uint64_t qfull, drain;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 E4M3 codes (one uint4) times one scale -> 8 BF16 pairs.
__device__ __forceinline__ void dequant16(uint4 c, float s, uint32_t* o) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    o[2 * i] = pack_bf16x2(f01.x * s, f01.y * s);
    o[2 * i + 1] = pack_bf16x2(f23.x * s, f23.y * s);
  }
}

__global__ void __launch_bounds__(kMlaThreads, 1) sparse_mla_kernel(const __grid_constant__ MlaParams p) {
  extern __shared__ __align__(1024) unsigned char mla_smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(mla_smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;                                   // kMlaStages x 73,728 B
  unsigned char* raw = base + kMlaStages * kMlaStageBytes;        // kMlaRawStages x 20,992 B
  MlaSmem* sm = reinterpret_cast<MlaSmem*>(raw + kMlaRawStages * kMlaRawBytes);
  const uint32_t stage_s = smem_u32(stages);
  const uint32_t raw_s = smem_u32(raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x / kMlaQuarters, qd = blockIdx.x % kMlaQuarters;
  const int r = find_request(p.qsl, p.R, t);
  const int seq_len = __ldg(p.seq_lens + r);

  // ---- set-up: barriers, tensor memory, the compacted top-k row
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMlaStages; ++i) {
      mbar_init(smem_u32(&sm->kfull[i]), kMlaProducers);
      mbar_init(smem_u32(&sm->kempty[i]), 1);
    }
    for (int i = 0; i < kMlaRawStages; ++i) {
      mbar_init(smem_u32(&sm->rfull[i]), 1);
      mbar_init(smem_u32(&sm->rempty[i]), 1);
    }
    mbar_init(smem_u32(&sm->sfull), 1);
    mbar_init(smem_u32(&sm->sfree), 128);
    mbar_init(smem_u32(&sm->pfull), 128);
    mbar_init(smem_u32(&sm->pvdone), 1);
    mbar_init(smem_u32(&sm->qfull), 128);
    mbar_init(smem_u32(&sm->drain), 1);
    sm->abort = 0;
    sm->conv_fail = 0;
    fence_barrier_init();
  }
  if (warp == kMlaMmaWarp) {
    tmem_alloc(smem_u32(&sm->tmem_base), 512);
    tmem_relinquish();
  }
  if (warp >= kMlaSoftmaxWarps && warp < kMlaMmaWarp) {
    // compaction: entries >= 0 in row order (entries beyond the context are
    // dropped), each resolved through the block table to its slot here, all
    // lookups in flight at once, so the loader's loop never waits on memory
    const int pt = threadIdx.x - kMlaSoftmaxWarps * 32;
    const int32_t* bt_row = p.block_table + (int64_t)r * p.max_blocks;
    const int per = (p.k + kMlaProducers - 1) / kMlaProducers;
    const int32_t* row = p.topk + (int64_t)t * p.k;
    int cnt = 0;
    bool bad = false;
    for (int i = 0; i < per; ++i) {
      const int j = pt * per + i;
      if (j < p.k) {
        const int e = __ldg(row + j);
        bad |= e >= seq_len;
        cnt += (e >= 0 && e < seq_len) ? 1 : 0;
      }
    }
    if (bad) raise_status(p.status, kStatusBadMetadata);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sm->warp_count[warp - kMlaSoftmaxWarps] = incl;
    named_bar_sync(1, kMlaProducers);
    int off = incl - cnt;
    for (int w = 0; w < warp - kMlaSoftmaxWarps; ++w) off += sm->warp_count[w];
    for (int i = 0; i < per; ++i) {
      const int j = pt * per + i;
      if (j < p.k) {
        const int e = __ldg(row + j);
        if (e >= 0 && e < seq_len) {
          const int blk = e / kPageTokens;
          const int64_t page = blk < p.max_blocks ? (int64_t)__ldg(bt_row + blk) : -1;
          const bool good = page >= 0 && page < p.num_pages;
          if (!good) raise_status(p.status, kStatusBadPage);
          sm->slot[off++] = good ? (int32_t)(page * kPageTokens + e % kPageTokens) : -1;
        }
      }
    }
    if (pt == kMlaProducers - 1) sm->n_valid = off;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const int n_valid = sm->n_valid;
  const int n_tiles = (n_valid + kMlaTile - 1) / kMlaTile;
  const int n_halves = (n_valid + kMlaHalf - 1) / kMlaHalf;
  volatile int* abort_flag = &sm->abort;

  if (warp < kMlaSoftmaxWarps) {
    // ================================================================ softmax
    const int h = threadIdx.x;  // head = tensor-memory lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const bool head_ok = h < p.Hq;
    // waits are taken warp-uniformly: the tensor-memory loads and stores that
    // follow them are warp-collective
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool ok = mbar_wait(smem_u32(bar), parity, abort_flag);
      return __all_sync(0xffffffffu, ok);
    };
    // queries into tensor memory (zero rows for heads beyond Hq)
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)t * p.Hq + h) * kMlaDim);
      for (int c = 0; c < 9; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = head_ok ? __ldg(src + c * 8 + u) : make_uint4(0u, 0u, 0u, 0u);
          w[4 * u] = v.x; w[4 * u + 1] = v.y; w[4 * u + 2] = v.z; w[4 * u + 3] = v.w;
        }
        tmem_st<32>(lane_base + kMlaColQ + 32 * c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->qfull));
    }
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    for (int i = 0; i < n_tiles && ok; ++i) {
      const uint32_t ph = (uint32_t)(i & 1);
      if (!wwait(&sm->sfull, ph)) { ok = false; break; }
      tc_fence_after();
      float x[64];
      {
        uint32_t sv[32];
        tmem_ld<32>(lane_base + kMlaColS, sv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(sv[j]);
        tmem_ld<32>(lane_base + kMlaColS + 32, sv);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) x[32 + j] = __uint_as_float(sv[j]);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->sfree));  // the next QK^T may overwrite the score tile
      const int left = n_valid - i * kMlaTile;  // valid tokens of this tile
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = j < left ? x[j] * p.scale_log2 : -INFINITY;
      // maximum as a tree (the four softmax warps are one per scheduler:
      // nothing hides a 64-long dependent chain)
      float mx[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) mx[j] = fmaxf(fmaxf(x[j], x[j + 16]), fmaxf(x[j + 32], x[j + 48]));
#pragma unroll
      for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) mx[j] = fmaxf(mx[j], mx[j + w]);
      const float mt = mx[0];
      // the previous PV has read the probability tile and written the output
      if (i > 0 && !wwait(&sm->pvdone, (uint32_t)((i - 1) & 1))) { ok = false; break; }
      tc_fence_after();
      const bool grow = mt > m_run + kMlaRescaleLog2;
      const float m_new = grow ? mt : m_run;
      if (__any_sync(0xffffffffu, grow && i > 0)) {
        const float alpha = (grow && i > 0) ? exp2f(m_run - m_new) : 1.0f;
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          tmem_ld<32>(lane_base + kMlaColO + 32 * c, ov);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
          tmem_st<32>(lane_base + kMlaColO + 32 * c, ov);
        }
        l_run *= alpha;
      }
      m_run = m_new;
      uint32_t pw[32];
      float ls[8];  // the sum of the probabilities the MMA multiplies, in 8 partial sums
#pragma unroll
      for (int j = 0; j < 8; ++j) ls[j] = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        pw[j] = pack_bf16x2(exp2f(x[2 * j] - m_run), exp2f(x[2 * j + 1] - m_run));
        const float2 pf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pw[j]));
        ls[j & 7] += pf.x + pf.y;
      }
      l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      tmem_st<32>(lane_base + kMlaColP, pw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->pfull));
    }
    if (ok && n_tiles > 0 && !wwait(&sm->pvdone, (uint32_t)((n_tiles - 1) & 1))) ok = false;
    if (!ok) {
      sm->abort = 1;
      raise_status(p.status, kStatusTimeout);
    } else {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.0f;
      uint16_t* orow = p.out + ((int64_t)t * p.Hq + h) * kMlaLatent + qd * 128;
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        if (n_tiles > 0) {
          tmem_ld<32>(lane_base + kMlaColO + 32 * c, ov);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          w[j] = pack_bf16x2(__uint_as_float(ov[2 * j]) * inv, __uint_as_float(ov[2 * j + 1]) * inv);
        if (head_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
      if (head_ok && qd == 0 && p.lse)
        p.lse[(int64_t)t * p.Hq + h] =
            l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }
  } else if (warp < kMlaMmaWarp) {
    // ================================================================ converters
    const int pt = threadIdx.x - kMlaSoftmaxWarps * 32;
    // Every converter reaches every named barrier, also after a wait gave up:
    // a failure is published in conv_fail and acted on, by all of them at
    // once, after the barrier.
    bool ok = true;
    for (int i = 0; i < n_tiles && ok; ++i) {
      const int b = i % kMlaStages;
      bool good = i < kMlaStages ||
                  mbar_wait(smem_u32(&sm->kempty[b]), (uint32_t)((i / kMlaStages - 1) & 1), abort_flag);
      const uint32_t sbase = stage_s + (uint32_t)(b * kMlaStageBytes);
      for (int hf = 0; hf < 2; ++hf) {
        const int g = 2 * i + hf;  // half tile
        const int rb = g % kMlaRawStages;
        const bool got = good && (g >= n_halves ||
                                  mbar_wait(smem_u32(&sm->rfull[rb]),
                                            (uint32_t)((g / kMlaRawStages) & 1), abort_flag));
        if (!got) sm->conv_fail = 1;
        const uint32_t live = (got && g < n_halves) ? sm->raw_live[rb] : 0u;
        const uint32_t rbase = raw_s + (uint32_t)(rb * kMlaRawBytes);
        // 32 tokens x 36 sixteen-element pieces; piece (n, cc) holds elements [16 cc, 16 cc + 16)
#pragma unroll
        for (int u = 0; u < (kMlaHalf * 36 + kMlaProducers - 1) / kMlaProducers; ++u) {
          const int job = pt + kMlaProducers * u;
          if (job < kMlaHalf * 36) {
            const int n = job / 36, cc = job - n * 36;
            uint32_t o[8];
            if ((live >> n) & 1u) {
              const uint32_t rec = rbase + (uint32_t)(n * kMlaRecBytes);
              dequant16(lds_v4(rec + 16u * (uint32_t)cc),
                        __uint_as_float(lds_u32(rec + (uint32_t)kMlaDim + 4u * (uint32_t)(cc >> 1))), o);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) o[j] = 0u;
            }
            // element 16 cc + j of tile row nn: chunk cc / 4, 16-byte units 2 (cc % 4) and +1
            const int nn = hf * kMlaHalf + n;
            const uint32_t row = sbase + (uint32_t)((cc >> 2) * kMlaChunkBytes + nn * 128);
            const uint32_t u0 = (uint32_t)(2 * (cc & 3));
            sts_v4(row + (((u0) ^ (uint32_t)(nn & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
            sts_v4(row + (((u0 + 1) ^ (uint32_t)(nn & 7)) << 4), make_uint4(o[4], o[5], o[6], o[7]));
          }
        }
        named_bar_sync(2, kMlaProducers);  // every converter is done with raw slot rb
        good = sm->conv_fail == 0;
        // the slot may be refilled (its reads are complete)
        if (pt == 0 && g < n_halves && good) mbar_arrive(smem_u32(&sm->rempty[rb]));
      }
      if (!good) { ok = false; break; }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&sm->kfull[b]));
    }
    if (!ok) sm->abort = 1;
  } else if (warp == kMlaLoaderWarp) {
    // ================================================================ loader
    // One bulk copy per selected record of the half tile, by the lane that
    // holds its slot.
    bool ok = true;
    int issued = 0;
    for (int g = 0; g < n_halves && ok; ++g) {
      const int rb = g % kMlaRawStages;
      if (g >= kMlaRawStages) {
        const bool got = mbar_wait(smem_u32(&sm->rempty[rb]),
                                   (uint32_t)((g / kMlaRawStages - 1) & 1), abort_flag);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      }
      const int ti = g * kMlaHalf + lane;
      const int sl = ti < n_valid ? sm->slot[ti] : -1;
      const uint32_t live = __ballot_sync(0xffffffffu, sl >= 0);
      const uint32_t bar = smem_u32(&sm->rfull[rb]);
      if (lane == 0) {
        sm->raw_live[rb] = live;
        mbar_arrive_expect_tx(bar, (uint32_t)__popc(live) * (uint32_t)kMlaRecBytes);
      }
      __syncwarp();
      if (sl >= 0)
        bulk_load(raw_s + (uint32_t)(rb * kMlaRawBytes + lane * kMlaRecBytes),
                  p.cache + (int64_t)(sl / kPageTokens) * kMlaPageBytes +
                      (int64_t)(sl % kPageTokens) * kMlaRecBytes,
                  (uint32_t)kMlaRecBytes, bar);
      issued = g + 1;
    }
    if (!ok) sm->abort = 1;
    // the latest phase of every raw slot this CTA expected has landed
    for (int j = issued > kMlaRawStages ? issued - kMlaRawStages : 0; j < issued; ++j)
      mbar_wait(smem_u32(&sm->rfull[j % kMlaRawStages]), (uint32_t)((j / kMlaRawStages) & 1), nullptr);
  } else if (lane == 0) {
    // ================================================================ MMA issuer
    const uint32_t id_qk = idesc_bf16_f32(128, kMlaTile, false);
    const uint32_t id_pv = idesc_bf16_f32(128, 128, true);
    bool ok = n_tiles == 0 || mbar_wait(smem_u32(&sm->qfull), 0, abort_flag);
    auto qk = [&](int i) -> bool {  // S = Q K_i^T, 36 instructions back to back
      const int st = i % kMlaStages;
      if (!mbar_wait(smem_u32(&sm->kfull[st]), (uint32_t)((i / kMlaStages) & 1), abort_flag)) return false;
      if (i > 0 && !mbar_wait(smem_u32(&sm->sfree), (uint32_t)((i - 1) & 1), abort_flag)) return false;
      tc_fence_after();
      const uint64_t d0 = sw128_desc(stage_s + (uint32_t)(st * kMlaStageBytes));
#pragma unroll
      for (int s = 0; s < kMlaDim / 16; ++s)
        umma_f16_ta(tmem + kMlaColS, tmem + kMlaColQ + 8 * s,
                    d0 + (uint64_t)(((s >> 2) * kMlaChunkBytes + (s & 3) * 32) >> 4), id_qk,
                    s > 0 ? 1u : 0u);
      umma_commit(smem_u32(&sm->sfull));
      return true;
    };
    auto pv = [&](int j) -> bool {  // O += P_j V_j
      const int st = j % kMlaStages;
      if (!mbar_wait(smem_u32(&sm->pfull), (uint32_t)(j & 1), abort_flag)) return false;
      tc_fence_after();
      const uint64_t v0 = sw128_desc_mn(stage_s + (uint32_t)(st * kMlaStageBytes + (2 * qd) * kMlaChunkBytes),
                                        kMlaChunkBytes, 1024);
#pragma unroll
      for (int kk = 0; kk < kMlaTile / 16; ++kk)
        umma_f16_ta(tmem + kMlaColO, tmem + kMlaColP + 8 * kk, v0 + (uint64_t)((kk * 16 * 128) >> 4),
                    id_pv, (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit(smem_u32(&sm->pvdone));
      umma_commit(smem_u32(&sm->kempty[st]));
      return true;
    };
    // PV of tile i-1 goes first: it releases tile i-1's stage to the
    // converters as soon as its probabilities are ready (measured faster than
    // issuing QK^T of tile i first, or interleaving the two).
    if (ok && n_tiles > 0) ok = qk(0);
    for (int i = 1; i < n_tiles && ok; ++i) {
      if (!pv(i - 1) || !qk(i)) ok = false;
    }
    if (ok && n_tiles > 0 && !pv(n_tiles - 1)) ok = false;
    // every MMA issued has completed before tensor memory is released
    umma_commit(smem_u32(&sm->drain));
    if (!mbar_wait(smem_u32(&sm->drain), 0, nullptr)) ok = false;
    if (!ok) {
      sm->abort = 1;
      raise_status(p.status, kStatusTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // After a wait gave up, copies issued before it may still be landing in
  // this CTA's shared memory (the loader's own drain waits are bounded too):
  // wait ~100 us for them before the CTA leaves.
  if (sm->abort)
    for (int k = 0; k < 100; ++k) __nanosleep(1000);
  if (warp == kMlaMmaWarp) tmem_dealloc(tmem, 512);
}

// Dynamic shared memory of the attention kernel (plus 1 KB for alignment).
constexpr size_t kMlaSmemBytes =
    (size_t)kMlaStages * kMlaStageBytes + (size_t)kMlaRawStages * kMlaRawBytes + sizeof(MlaSmem) + 1024;

}  // namespace dsa
