// Vocabulary sorting of Cut Cross-Entropy (Sec. 4.3, "Vocabulary sorting"):
// the backward visits the vocabulary in order of decreasing average logit, so
// ids of similar average share a 256-id block and the gradient filter finds
// more blocks it can leave out.
//
// The average logit of id v over the valid rows is
//     a_v = (1/count) sum_{valid n} (H_n . W_v + b_v) = W_v . mean_valid(H) + b_v,
// so it costs one pass over H (column sums) and one over W (a matrix-vector
// product), not an atomic update per logit tile as in the paper's forward.
// Every sum runs in a fixed order, so the order is bit-reproducible.
//
//   hsum_partial_kernel   column sums of H over the valid rows, per row split
//   hmean_kernel          fixed-order sum of the splits / count
//   avg_logit_kernel      a_v in fp32, and a 32-bit key whose ascending order
//                         is the descending order of a_v
//   radix_*_kernel        stable LSD radix sort of the keys
//   gather_vocab_kernel   W and the bias rearranged in the sorted order
//   remap_targets_kernel  each target replaced by its sorted position
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace flce {

constexpr int kHsumMaxSplits = 256;    // row splits of the column sums
constexpr int kHsumRowsPerSplit = 32;  // fewest rows a split gets before splits are added
constexpr int kHsumCols = 2048;        // columns per block: 8 per thread
constexpr int kVocabWarpsPerBlock = 8;

__device__ __forceinline__ bool sort_target_valid(int64_t t, int64_t vocab, int64_t ignore_index) {
  return t != ignore_index && t >= 0 && t < vocab;
}

__host__ __device__ inline int hsum_splits(int64_t n) {
  const int64_t s = (n + kHsumRowsPerSplit - 1) / kHsumRowsPerSplit;
  return (int)(s < 1 ? 1 : (s > kHsumMaxSplits ? kHsumMaxSplits : s));
}

// part[s][c] = sum of H[r][c] over the valid rows r of split s, in ascending
// row order. Block (x, s) covers columns x*2048 .. x*2048+2047, eight per
// thread (one 16-byte load per row); d is a multiple of 8.
__global__ void __launch_bounds__(256) hsum_partial_kernel(const __nv_bfloat16* __restrict__ H, int64_t n, int d,
                                                           const int64_t* __restrict__ y, int64_t vocab,
                                                           int64_t ignore_index, int splits,
                                                           float* __restrict__ part) {
  const int c = blockIdx.x * kHsumCols + threadIdx.x * 8;
  const int s = blockIdx.y;
  const int64_t per = (n + splits - 1) / splits;
  const int64_t r0 = (int64_t)s * per, r1 = min(n, r0 + per);
  if (c >= d) return;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll 4
  for (int64_t r = r0; r < r1; ++r) {
    const float m = sort_target_valid(__ldg(y + r), vocab, ignore_index) ? 1.f : 0.f;
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(H + r * d + c));
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h2[j]);
      acc[2 * j] = fmaf(m, f.x, acc[2 * j]);
      acc[2 * j + 1] = fmaf(m, f.y, acc[2 * j + 1]);
    }
  }
  float4* out = reinterpret_cast<float4*>(part + (size_t)s * d + c);
  out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// mean[c] = (part[0][c] + part[1][c] + ... in split order) / count; all zero
// when no row is valid.
__global__ void hmean_kernel(const float* __restrict__ part, int splits, int d, const int64_t* __restrict__ count,
                             float* __restrict__ mean) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  float t = 0.f;
  for (int s = 0; s < splits; ++s) t += part[(size_t)s * d + c];
  const int64_t cnt = *count;
  mean[c] = cnt > 0 ? t / (float)cnt : 0.f;
}

// Ascending order of the returned key is descending order of x (with -0
// taken as +0 by the caller): flip every bit of a negative value, set the
// sign bit of a non-negative one, then complement.
__device__ __forceinline__ uint32_t descending_key(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ~asc;
}

// avg[v] = W_v . mean (+ bias[v]) and key[v] = descending_key(avg[v]). One
// warp per vocabulary row: lane l takes the 8-element groups l, l + 32, ...
// of the row in order, and lane 0 keeps the sum of a fixed butterfly.
__global__ void __launch_bounds__(kVocabWarpsPerBlock * 32) avg_logit_kernel(
    const __nv_bfloat16* __restrict__ W, int64_t vocab, int d, const float* __restrict__ mean,
    const float* __restrict__ bias, float* __restrict__ avg, uint32_t* __restrict__ key) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * kVocabWarpsPerBlock;
  const int groups = d / 8;
  const float4* m4 = reinterpret_cast<const float4*>(mean);
  for (int64_t v = (int64_t)blockIdx.x * kVocabWarpsPerBlock + (threadIdx.x >> 5); v < vocab; v += warps) {
    const uint4* row = reinterpret_cast<const uint4*>(W + v * d);
    float acc = 0.f;
    for (int g = lane; g < groups; g += 32) {
      const uint4 q = __ldg(row + g);
      const float4 a = __ldg(m4 + 2 * g), b = __ldg(m4 + 2 * g + 1);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&q);
      const float2 w0 = __bfloat1622float2(h2[0]), w1 = __bfloat1622float2(h2[1]);
      const float2 w2 = __bfloat1622float2(h2[2]), w3 = __bfloat1622float2(h2[3]);
      acc = fmaf(w0.x, a.x, acc);
      acc = fmaf(w0.y, a.y, acc);
      acc = fmaf(w1.x, a.z, acc);
      acc = fmaf(w1.y, a.w, acc);
      acc = fmaf(w2.x, b.x, acc);
      acc = fmaf(w2.y, b.y, acc);
      acc = fmaf(w3.x, b.z, acc);
      acc = fmaf(w3.y, b.w, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      float x = acc + (bias ? __ldg(bias + v) : 0.f);
      if (x == 0.f) x = 0.f;   // one key for +0 and -0
      avg[v] = x;
      key[v] = descending_key(x);
    }
  }
}

// Stable LSD radix sort of n 32-bit keys with their ids: 8-bit digits, four
// passes, each of three launches over tiles of kSortTile keys (one block per
// tile). For pass `shift`:
//   radix_hist_kernel     digit counts of every tile, hist[d * tiles + b];
//   radix_scan_kernel     exclusive prefix sums of hist in that (digit-major,
//                         tile-minor) order: where tile b's keys of digit d go;
//   radix_scatter_kernel  each key to that offset plus its rank among the
//                         tile's keys of the same digit, counted in tile order.
// Ranks keep the input order of equal digits, so every pass is stable and the
// output positions are a permutation of [0, n). radix_inverse_kernel then
// writes inv[ids[i]] = i.
constexpr int kSortTile = 4096;
constexpr int kSortWarpsPerTile = 8;                      // 256 threads
constexpr int kSortWarpKeys = kSortTile / kSortWarpsPerTile;

__global__ void __launch_bounds__(256) radix_hist_kernel(const uint32_t* __restrict__ keys, int n, int shift,
                                                         uint32_t* __restrict__ hist) {
  __shared__ uint32_t cnt[256];
  const int b = blockIdx.x, lane = threadIdx.x & 31;
  cnt[threadIdx.x] = 0u;
  __syncthreads();
  const int t0 = b * kSortTile, t1 = min(n, t0 + kSortTile);
  for (int base = t0; base < t1; base += 256) {
    const int i = base + threadIdx.x;
    const bool act = i < t1;
    const unsigned mask = __ballot_sync(0xffffffffu, act);
    if (act) {
      const uint32_t d = (keys[i] >> shift) & 255u;
      const unsigned peers = __match_any_sync(mask, d);
      if ((peers & ((1u << lane) - 1u)) == 0u) atomicAdd(&cnt[d], (uint32_t)__popc(peers));
    }
  }
  __syncthreads();
  hist[(size_t)threadIdx.x * gridDim.x + b] = cnt[threadIdx.x];
}

__global__ void __launch_bounds__(1024) radix_scan_kernel(uint32_t* __restrict__ hist, int count) {
  __shared__ uint32_t part[1024];
  const int per = (count + 1023) / 1024;
  const int s0 = min(count, (int)threadIdx.x * per), s1 = min(count, s0 + per);
  uint32_t sum = 0u;
  for (int i = s0; i < s1; ++i) sum += hist[i];
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const uint32_t v = threadIdx.x >= (unsigned)o ? part[threadIdx.x - o] : 0u;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  uint32_t run = threadIdx.x ? part[threadIdx.x - 1] : 0u;
  for (int i = s0; i < s1; ++i) {
    const uint32_t c = hist[i];
    hist[i] = run;
    run += c;
  }
}

// Warp w of the block takes keys [w * 512, (w + 1) * 512) of the tile in
// chunks of 32: first it counts its digits, then each key's output position
// is the tile's offset for the digit, plus the counts of earlier warps, plus
// the warp's running count, plus the key's rank among lower lanes of its
// chunk with the same digit. ids_in == nullptr means ids 0..n-1.
__global__ void __launch_bounds__(256) radix_scatter_kernel(const uint32_t* __restrict__ keys_in,
                                                            const int32_t* __restrict__ ids_in, int n, int shift,
                                                            const uint32_t* __restrict__ offs,
                                                            uint32_t* __restrict__ keys_out,
                                                            int32_t* __restrict__ ids_out) {
  __shared__ uint32_t wpos[kSortWarpsPerTile][256];
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = b * kSortTile, t1 = min(n, t0 + kSortTile);
  const int w0 = min(t1, t0 + warp * kSortWarpKeys), w1 = min(t1, w0 + kSortWarpKeys);
  const unsigned below = (1u << lane) - 1u;
  for (int i = threadIdx.x; i < kSortWarpsPerTile * 256; i += 256) (&wpos[0][0])[i] = 0u;
  __syncthreads();
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool act = i < w1;
    const unsigned mask = __ballot_sync(0xffffffffu, act);
    if (act) {
      const uint32_t d = (keys_in[i] >> shift) & 255u;
      const unsigned peers = __match_any_sync(mask, d);
      if ((peers & below) == 0u) wpos[warp][d] += (uint32_t)__popc(peers);
    }
    __syncwarp();
  }
  __syncthreads();
  {
    const int d = threadIdx.x;
    uint32_t run = offs[(size_t)d * gridDim.x + b];
    for (int w = 0; w < kSortWarpsPerTile; ++w) {
      const uint32_t c = wpos[w][d];
      wpos[w][d] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool act = i < w1;
    const unsigned mask = __ballot_sync(0xffffffffu, act);
    if (act) {
      const uint32_t k = keys_in[i];
      const int32_t id = ids_in ? ids_in[i] : i;
      const uint32_t d = (k >> shift) & 255u;
      const unsigned peers = __match_any_sync(mask, d);
      const uint32_t rank = (uint32_t)__popc(peers & below);
      const uint32_t pos = wpos[warp][d] + rank;
      keys_out[pos] = k;
      ids_out[pos] = id;
      __syncwarp(mask);
      if (rank == 0u) wpos[warp][d] += (uint32_t)__popc(peers);
    }
    __syncwarp();
  }
}

__global__ void radix_inverse_kernel(const int32_t* __restrict__ ids, int n, int32_t* __restrict__ inv) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) inv[ids[i]] = i;
}

// Ws[i] = W[order[i]] (rows of row_vec 16-byte groups) and, with a bias,
// bias_s[i] = bias[order[i]]. One warp per row; order is a permutation of
// [0, vocab).
__global__ void __launch_bounds__(kVocabWarpsPerBlock * 32) gather_vocab_kernel(
    const uint4* __restrict__ W, int row_vec, const int32_t* __restrict__ order, int64_t vocab,
    uint4* __restrict__ Ws, const float* __restrict__ bias, float* __restrict__ bias_s) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * kVocabWarpsPerBlock;
  for (int64_t i = (int64_t)blockIdx.x * kVocabWarpsPerBlock + (threadIdx.x >> 5); i < vocab; i += warps) {
    const int64_t src = __ldg(order + i);
    const uint4* from = W + src * row_vec;
    uint4* to = Ws + i * row_vec;
    for (int k = lane; k < row_vec; k += 32) to[k] = __ldg(from + k);
    if (bias && lane == 0) bias_s[i] = __ldg(bias + src);
  }
}

// ys[n] = sorted position of target y[n]; -1 (which the sorted backward
// takes as its ignore index) for ignored and out-of-range targets.
__global__ void remap_targets_kernel(const int64_t* __restrict__ y, int64_t n, int64_t vocab, int64_t ignore_index,
                                     const int32_t* __restrict__ inv, int64_t* __restrict__ ys) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n) return;
  const int64_t t = y[r];
  ys[r] = sort_target_valid(t, vocab, ignore_index) ? (int64_t)__ldg(inv + t) : -1;
}

}  // namespace flce
