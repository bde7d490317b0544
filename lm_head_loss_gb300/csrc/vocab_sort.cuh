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
//   radix_sort_kernel     stable LSD radix sort of the keys (one block)
//   gather_vocab_kernel   W and the bias rearranged in the sorted order
//   remap_targets_kernel  each target replaced by its sorted position
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace flce {

constexpr int kHsumMaxSplits = 256;    // row splits of the column sums
constexpr int kHsumRowsPerSplit = 32;  // fewest rows a split gets before splits are added
constexpr int kHsumCols = 2048;        // columns per block: 8 per thread
constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortBatch = 8;          // keys a lane loads ahead in the scatter
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

// Stable LSD radix sort of n 32-bit keys, 8-bit digits, four passes, in one
// block of 32 warps. Warp w owns the contiguous segment w of the array. Each
// pass counts every warp's digits, turns the counts into an output offset per
// (digit, warp) in digit-major, warp-minor order, and scatters each warp's
// segment in its original order (ranks among equal digits from
// __match_any_sync), so equal digits keep their relative order and the
// output positions form a permutation of [0, n). ids start as 0..n-1. On
// return keys_a/ids_a hold the sorted keys and ids and inv[ids_a[i]] = i.
__global__ void __launch_bounds__(kSortThreads, 1) radix_sort_kernel(uint32_t* __restrict__ keys_a,
                                                                    uint32_t* __restrict__ keys_b,
                                                                    int32_t* __restrict__ ids_a,
                                                                    int32_t* __restrict__ ids_b,
                                                                    int32_t* __restrict__ inv, int n) {
  __shared__ uint32_t offs[kSortWarps][256];
  __shared__ uint32_t digit_base[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = (int)(((int64_t)n + kSortWarps - 1) / kSortWarps);
  const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
  uint32_t* kin = keys_a;
  uint32_t* kout = keys_b;
  int32_t* iin = ids_a;
  int32_t* iout = ids_b;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = pass * 8;
    for (int i = threadIdx.x; i < kSortWarps * 256; i += kSortThreads) (&offs[0][0])[i] = 0u;
    __syncthreads();
#pragma unroll 4
    for (int i = s0 + lane; i < s1; i += 32) atomicAdd(&offs[warp][(kin[i] >> shift) & 255u], 1u);
    __syncthreads();
    if (threadIdx.x < 256) {
      const int dg = threadIdx.x;
      uint32_t run = 0;
      for (int w = 0; w < kSortWarps; ++w) {
        const uint32_t c = offs[w][dg];
        offs[w][dg] = run;
        run += c;
      }
      digit_base[dg] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t run = 0;
      for (int dg = 0; dg < 256; ++dg) {
        const uint32_t c = digit_base[dg];
        digit_base[dg] = run;
        run += c;
      }
    }
    __syncthreads();
    if (threadIdx.x < 256)
      for (int w = 0; w < kSortWarps; ++w) offs[w][threadIdx.x] += digit_base[threadIdx.x];
    __syncthreads();
#pragma unroll 1
    for (int base = s0; base < s1; base += 32 * kSortBatch) {
      uint32_t kk[kSortBatch];
      int32_t ii[kSortBatch];
#pragma unroll
      for (int b = 0; b < kSortBatch; ++b) {
        const int i = base + b * 32 + lane;
        kk[b] = i < s1 ? kin[i] : 0u;
        ii[b] = i < s1 ? (pass == 0 ? i : iin[i]) : 0;
      }
#pragma unroll
      for (int b = 0; b < kSortBatch; ++b) {
        const int i = base + b * 32 + lane;
        const bool act = i < s1;
        const unsigned mask = __ballot_sync(0xffffffffu, act);
        if (act) {
          const uint32_t dg = (kk[b] >> shift) & 255u;
          const unsigned peers = __match_any_sync(mask, dg);
          const int rank = __popc(peers & ((1u << lane) - 1u));
          const uint32_t pos = offs[warp][dg] + (uint32_t)rank;
          kout[pos] = kk[b];
          iout[pos] = ii[b];
          __syncwarp(mask);
          if (rank == 0) offs[warp][dg] += (uint32_t)__popc(peers);
        }
        __syncwarp();
      }
    }
    __syncthreads();
    uint32_t* tk = kin;
    kin = kout;
    kout = tk;
    int32_t* ti = iin;
    iin = iout;
    iout = ti;
  }
  for (int i = threadIdx.x; i < n; i += kSortThreads) inv[iin[i]] = i;
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
