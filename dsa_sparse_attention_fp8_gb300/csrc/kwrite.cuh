// Indexer-key cache write (slot mapping + per-block FP8 quantisation) and the
// stand-alone block quantiser.
//
// "GLM-5.3 推理全链路(十二)", write-path section: every F layer stores each new
// token's FP8 key and FP32 scale at the token's in-page offset; byte-accounting
// table: 128 E4M3 bytes + one FP32 scale = 132 B per token.  "HBM 索引架构设计"
// §2.3: slot = block_table[req, pos / 64] * 64 + pos % 64.
//
// One warp per 128-element block: each lane owns 4 consecutive elements
// (one float4 load), the block's absolute maximum comes from a warp
// reduction, and every lane writes its 4 code bytes as one 32-bit store, so a
// warp writes the 128-byte key row in one coalesced transaction.
#pragma once

#include <cuda_fp8.h>
#include <cstdint>

#include "ptx.cuh"

namespace dsa {

constexpr int kHeadDim = 128;
constexpr int kPageTokens = 64;
constexpr int kPageBytes = 8448;
constexpr int kPageScaleOffset = 8192;

constexpr int kStatusBadPage = 0x1;
constexpr int kStatusBadMetadata = 0x2;
constexpr int kStatusTimeout = 0x4;

__device__ __forceinline__ void raise_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Quantise this lane's 4 elements of a 128-element block.  Returns the 4 E4M3
// codes packed little-endian (element 4*lane first) and the block scale.
// s = amax / 448 (IEEE FP32 division), s = 1 for an all-zero block; each code
// is E4M3(x / s), round-to-nearest-even, saturating.
__device__ __forceinline__ uint32_t quantize_lane4(float4 v, float* scale_out) {
  float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float s = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
  float2 lo = make_float2(__fdiv_rn(v.x, s), __fdiv_rn(v.y, s));
  float2 hi = make_float2(__fdiv_rn(v.z, s), __fdiv_rn(v.w, s));
  uint32_t c01 = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
  uint32_t c23 = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
  *scale_out = s;
  return (c01 & 0xFFFFu) | ((c23 & 0xFFFFu) << 16);
}

// Request that owns query row t: the last r with query_start_loc[r] <= t.
__device__ __forceinline__ int find_request(const int32_t* __restrict__ qsl, int R, int t) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The same search over a copy of query_start_loc in shared memory.
__device__ __forceinline__ int find_request_smem(const int32_t* qsl_s, int R, int t) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (qsl_s[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// query_start_loc entries staged in shared memory by the cache-write kernel
// (its binary search would otherwise be a chain of dependent global loads)
constexpr int kQslSmem = 4096;

// One lane's 4 consecutive elements of 128-element block `blk` as FP32
// (BF16 widens exactly: its bits are the upper half of the FP32 value).
__device__ __forceinline__ float4 load_lane4(const float* x, int64_t blk, int lane) {
  return __ldg(reinterpret_cast<const float4*>(x + blk * kHeadDim) + lane);
}
__device__ __forceinline__ float4 load_lane4(const uint16_t* x, int64_t blk, int lane) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(x + blk * kHeadDim) + lane);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

// Warps [0, T): the new tokens' keys (quantise, slot mapping, write into the
// page pool).  Warps [T, T + T*H) when q is given: the query rows' H blocks
// each, quantised to q_codes [T, H, 128] and q_scales [T, H] with the same
// rule, so one launch performs the whole per-token quantisation of a layer.
//
// Compressed cache ("HBM 索引架构设计" §5.2), ratio > 1: only a token with
// (pos + 1) % ratio == 0 holds an entry, number pos / ratio, stored through
// the block table like a token position; the others get slot -1 and write
// nothing.  ratio 1 is the plain cache.
template <typename TIn>
__global__ void __launch_bounds__(256) write_k_kernel(
    const TIn* __restrict__ k, int T, const int32_t* __restrict__ qsl,
    const int32_t* __restrict__ seq_lens, int R, const int32_t* __restrict__ block_table,
    int max_blocks, uint8_t* __restrict__ k_cache, int64_t num_pages, int ratio,
    int64_t* __restrict__ slot_mapping, int32_t* status, const TIn* __restrict__ q, int H,
    uint8_t* __restrict__ q_codes, float* __restrict__ q_scales) {
  pdl_launch_dependents();  // the scoring kernel's prologue may overlap this write
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  // the key's load is in flight while the block stages query_start_loc
  const float4 v = warp < T ? load_lane4(k, warp, lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  __shared__ int32_t qsl_s[kQslSmem];
  const bool staged = R + 1 <= kQslSmem;
  if (staged) {
    for (int i = threadIdx.x; i <= R; i += blockDim.x) qsl_s[i] = __ldg(qsl + i);
    __syncthreads();
  }
  if (warp >= T) {
    const int64_t b = warp - T;
    if (q == nullptr || b >= (int64_t)T * H) return;
    float s;
    const uint32_t c = quantize_lane4(load_lane4(q, b, lane), &s);
    reinterpret_cast<uint32_t*>(q_codes + b * kHeadDim)[lane] = c;
    if (lane == 0) q_scales[b] = s;
    return;
  }
  const int t = (int)warp;
  float s;
  const uint32_t codes = quantize_lane4(v, &s);

  const int r = staged ? find_request_smem(qsl_s, R, t) : find_request(qsl, R, t);
  const int q_begin = staged ? qsl_s[r] : __ldg(qsl + r);
  const int q_len = (staged ? qsl_s[r + 1] : __ldg(qsl + r + 1)) - q_begin;
  const int seq_len = __ldg(seq_lens + r);
  const int pos = seq_len - q_len + (t - q_begin);
  int64_t slot = -1;
  const int entry = pos / ratio;  // cache entry of a token that completes one
  if (q_len < 0 || seq_len < q_len || pos < 0 || pos >= seq_len ||
      ((pos + 1) % ratio == 0 && entry / kPageTokens >= max_blocks)) {
    if (lane == 0) raise_status(status, kStatusBadMetadata);
  } else if ((pos + 1) % ratio == 0) {
    const int64_t page = __ldg(block_table + (int64_t)r * max_blocks + entry / kPageTokens);
    if (page < 0 || page >= num_pages) {
      if (lane == 0) raise_status(status, kStatusBadPage);
    } else {
      const int off = entry % kPageTokens;
      uint8_t* pg = k_cache + page * kPageBytes;
      reinterpret_cast<uint32_t*>(pg + off * kHeadDim)[lane] = codes;
      if (lane == 0) *reinterpret_cast<float*>(pg + kPageScaleOffset + off * 4) = s;
      slot = page * kPageTokens + off;
    }
  }
  if (slot_mapping && lane == 0) slot_mapping[t] = slot;
}

__global__ void __launch_bounds__(256) quantize_blocks_kernel(const float* __restrict__ x,
                                                              int64_t n_blocks,
                                                              uint8_t* __restrict__ codes,
                                                              float* __restrict__ scales) {
  const int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= n_blocks) return;
  const float4 v = __ldg(reinterpret_cast<const float4*>(x + b * kHeadDim) + lane);
  float s;
  const uint32_t c = quantize_lane4(v, &s);
  reinterpret_cast<uint32_t*>(codes + b * kHeadDim)[lane] = c;
  if (lane == 0) scales[b] = s;
}

}  // namespace dsa
