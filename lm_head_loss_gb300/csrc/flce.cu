// C-ABI of the fused LM-head cross-entropy (declared in include/flce.h):
// argument checks, workspace layout, chunk schedule, TMA tensor maps, and the
// small reduction kernels around the tcgen05 GEMM of tile_gemm.cuh.
//
// Schedule of flce_forward_backward (every launch on the caller's stream):
//   prep                      validate targets, count valid rows, reset status
//   per row chunk (<= 8192 rows):
//     GEMM  EPI_LSE           logits tile -> per-tile (max, sum-exp) + target logit
//     lse_combine             fixed-order merge of the tile partials -> LSE, row losses
//   finalize                  fixed-order fp64 sum -> mean loss, scale = g / count
//   per row chunk, per vocabulary chunk (<= 10240 ids, picked by a makespan
//   model; dW and dH of chunk c run in one launch with EPI_DZ of chunk c+1):
//     GEMM  EPI_DZ            recomputed logits -> bf16 G = softmax - onehot -> staging
//     GEMM  dW chunk          dW[v-chunk] (=|+=) scale * staging^T H[row chunk]
//     GEMM  dH chunk          dH[row chunk] (=|+=) scale * staging W[v-chunk]
// The first contribution to an output tile is a plain store and later ones a
// TMA reduce-add, so no output needs zeroing and every sum runs in launch
// order: results are bit-reproducible.
//
// Options around that schedule: a bias and mean / sum / none reductions
// (flce_forward_ex, flce_backward_ex), the gradient filter's per-tile flags
// and keep masks, ignored-row compaction, vocabulary sorting
// (vocab_sort.cuh), and AdamW on W applied in the dW epilogue
// (flce_forward_backward_adamw) or after it (flce_adamw_step).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "flce.h"
#include "tile_gemm.cuh"
#include "tile_gemm_pair.cuh"
#include "vocab_sort.cuh"

namespace flce {

constexpr int kRowChunk = 8192;    // rows per chunk (multiple of 256)
constexpr int kVocabChunkMin = 4096;   // candidate vocabulary chunks of the backward (multiples of 256);
constexpr int kVocabChunkMax = 10240;  // the workspace is sized for the largest
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint64_t kShortWaitNs = 1000ull;

struct alignas(256) WsHeader {
  uint32_t status;
  uint32_t filter_on;
  int64_t count;
  float scale;
  float loss;
  unsigned long long tiles_total;
  unsigned long long tiles_skipped;
  float opt[kAdamwConsts];   // fused AdamW step constants (flce_forward_backward_adamw)
};
static_assert(sizeof(WsHeader) == 256, "the header occupies the first 256 bytes of the workspace");

// ------------------------------------------------------------------ kernels

// One block: count targets in [0, V), flag targets that are neither ignored
// nor in range, reset the status word and the filter statistics.
__global__ void prep_kernel(const int64_t* __restrict__ y, int64_t n, int64_t vocab, int64_t ignore_index,
                            uint32_t filter_on, WsHeader* hdr) {
  __shared__ long long s_cnt[32];
  __shared__ unsigned s_bad[32];
  long long cnt = 0;
  unsigned bad = 0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t t = y[i];
    if (t == ignore_index) continue;
    if (t >= 0 && t < vocab)
      ++cnt;
    else
      bad = 1u;
  }
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_down_sync(0xffffffffu, cnt, o);
    bad |= __shfl_down_sync(0xffffffffu, bad, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    s_cnt[w] = cnt;
    s_bad[w] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long c = 0;
    unsigned b = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      c += s_cnt[i];
      b |= s_bad[i];
    }
    hdr->count = c;
    hdr->status = b ? kDevBadTarget : 0u;
    hdr->filter_on = filter_on;
    hdr->tiles_total = 0ull;
    hdr->tiles_skipped = 0ull;
  }
}

// One block: the number of targets in [0, V) that are not ignore_index
// (the rows a mean counts), written to *count.
__global__ void count_valid_kernel(const int64_t* __restrict__ y, int64_t n, int64_t vocab, int64_t ignore_index,
                                   int64_t* __restrict__ count) {
  __shared__ long long s_cnt[32];
  long long cnt = 0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t t = y[i];
    cnt += (t != ignore_index && t >= 0 && t < vocab) ? 1 : 0;
  }
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_down_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) s_cnt[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long c = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) c += s_cnt[i];
    *count = c;
  }
}

// Merge of the per-tile (max, sum) partials into LSE_n. A block covers 32
// rows; thread (r, g) merges tiles g, g + 32, g + 64, ... of row r, then the
// 32 partials of a row are merged in g order and the 32 row losses of the
// block are summed in a fixed order (fp64). 1024 threads per block keep
// enough loads in flight to read the partials near HBM speed.
constexpr int kCombineRows = 32;
constexpr int kCombineSplit = 32;

__device__ __forceinline__ void lse_merge(float& mx, float& sm, float m, float s) {
  if (m > mx) {
    sm = sm * exp2f(mx - m) + s;
    mx = m;
  } else {
    sm += s * exp2f(m - mx);
  }
}

__global__ void __launch_bounds__(kCombineRows * kCombineSplit)
    lse_combine_kernel(const float* __restrict__ part_m, const float* __restrict__ part_s, int part_ld, int n_tiles,
                       const float* __restrict__ zy, const int64_t* __restrict__ y, int64_t row0, int rows,
                       int64_t vocab, int64_t ignore_index, float* __restrict__ lse_out,
                       double* __restrict__ block_sums, float* __restrict__ loss_rows) {
  __shared__ float sh_m[kCombineSplit][kCombineRows];
  __shared__ float sh_s[kCombineSplit][kCombineRows];
  __shared__ double red[kCombineRows];
  const int r = threadIdx.x, g = threadIdx.y;
  const int lr = blockIdx.x * kCombineRows + r;
  float mx = -INFINITY, sm = 0.f;
  if (lr < rows) {
    for (int t = g; t < n_tiles; t += kCombineSplit)
      lse_merge(mx, sm, part_m[(size_t)t * part_ld + lr], part_s[(size_t)t * part_ld + lr]);
  }
  sh_m[g][r] = mx;
  sh_s[g][r] = sm;
  __syncthreads();
  if (g == 0) {
    double contrib = 0.0;
    if (lr < rows) {
      for (int k = 1; k < kCombineSplit; ++k) lse_merge(mx, sm, sh_m[k][r], sh_s[k][r]);
      const float lse = (mx + log2f(sm)) * 0.69314718055994531f;
      lse_out[row0 + lr] = lse;
      const int64_t t = y[row0 + lr];
      if (t != ignore_index && t >= 0 && t < vocab) contrib = (double)lse - (double)zy[lr];
      if (loss_rows) loss_rows[row0 + lr] = (float)contrib;
    }
    red[r] = contrib;
  }
  __syncthreads();
  if (g == 0 && r == 0) {
    double acc = 0.0;
    for (int k = 0; k < kCombineRows; ++k) acc += red[k];
    block_sums[row0 / kCombineRows + blockIdx.x] = acc;
  }
}

// One block: fixed-order fp64 sum of the per-block row losses, mean over the
// valid count (clamped to one), and the gradient scale g / count.
// count_global (or NULL): the valid count of every rank of a data-parallel
// step, which replaces this call's own count in the mean.
__global__ void finalize_kernel(const double* __restrict__ block_sums, int n_blocks, float grad_loss, WsHeader* hdr,
                                float* loss_out, int reduction, const int64_t* __restrict__ count_global) {
  __shared__ double red[256];
  double acc = 0.0;
  for (int i = threadIdx.x; i < n_blocks; i += 256) acc += block_sums[i];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    // reduction 0 = mean over the valid count (clamped to 1), 1 = sum, 2 = none.
    // A forward whose GEMM gave up on a bounded wait has no valid partials:
    // its loss is NaN, so no caller mistakes it for a result.
    const int64_t count = count_global ? *count_global : hdr->count;
    const double denom = reduction == 0 ? (double)(count > 0 ? count : 1) : 1.0;
    const float loss = (hdr->status & kDevTimeout) ? __int_as_float(0x7fc00000) : (float)(red[0] / denom);
    hdr->loss = loss;
    hdr->scale = reduction == 2 ? 1.0f : (float)((double)grad_loss / denom);
    if (reduction != 2) *loss_out = loss;
  }
}

// Gradient scale of a backward whose upstream gradient lives on the device:
// g / max(count, 1) for a mean, g for a sum, 1 for per-row gradients (they
// scale G inside the dZ epilogue).
__global__ void set_scale_kernel(const float* __restrict__ grad, int reduction, WsHeader* hdr) {
  if (threadIdx.x == 0) {
    const double denom = reduction == 0 ? (double)(hdr->count > 0 ? hdr->count : 1) : 1.0;
    hdr->scale = reduction == 2 ? 1.0f : (float)((double)grad[0] / denom);
  }
}

// Constants of one fused AdamW step from the caller's device-side
// hyper-parameters, the bias corrections in fp64. A step below 1, or a beta
// outside [0, 1), records kDevBadHparams and turns the step into one that
// leaves the weights unchanged.
__global__ void adamw_prep_kernel(const flce_adamw_hparams* __restrict__ hp, WsHeader* hdr) {
  if (threadIdx.x != 0) return;
  const flce_adamw_hparams h = *hp;
  const bool ok = h.step >= 1 && h.beta1 >= 0.f && h.beta1 < 1.f && h.beta2 >= 0.f && h.beta2 < 1.f &&
                  h.eps > 0.f && isfinite(h.lr) && isfinite(h.weight_decay);
  if (!ok) {
    atomicOr(&hdr->status, kDevBadHparams);
    const float keep[kAdamwConsts] = {0.f, 1.f, 1.f, 1.f, 1.f, 1.f};
    for (int i = 0; i < kAdamwConsts; ++i) hdr->opt[i] = keep[i];
    return;
  }
  const double t = (double)h.step;
  const double bc1 = 1.0 - pow((double)h.beta1, t), bc2 = 1.0 - pow((double)h.beta2, t);
  hdr->opt[0] = (float)((double)h.lr / bc1);
  hdr->opt[1] = (float)(1.0 / sqrt(bc2));
  hdr->opt[2] = (float)(1.0 - (double)h.lr * (double)h.weight_decay);
  hdr->opt[3] = h.beta1;
  hdr->opt[4] = h.beta2;
  hdr->opt[5] = h.eps;
}

// One AdamW step on n elements (flce_adamw_step), with the constants of
// adamw_prep_kernel and the arithmetic of the fused EPI_ADAMW epilogue
// (adamw_update).
// Thread i takes elements 4i .. 4i+3 of the vector part (all pointers
// 16-byte aligned), then the last n % 4 elements one by one.
__global__ void __launch_bounds__(256) adamw_step_kernel(const WsHeader* __restrict__ hdr, const float* __restrict__ grad,
                                                         float* __restrict__ p, float* __restrict__ m,
                                                         float* __restrict__ v, __nv_bfloat16* __restrict__ w,
                                                         int64_t n) {
  float c[kAdamwConsts];
  for (int i = 0; i < kAdamwConsts; ++i) c[i] = hdr->opt[i];
  const int64_t n4 = n / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 g4 = reinterpret_cast<const float4*>(grad)[i];
    float4 p4 = reinterpret_cast<float4*>(p)[i], m4 = reinterpret_cast<float4*>(m)[i],
           v4 = reinterpret_cast<float4*>(v)[i];
    adamw_update(c, g4.x, p4.x, m4.x, v4.x);
    adamw_update(c, g4.y, p4.y, m4.y, v4.y);
    adamw_update(c, g4.z, p4.z, m4.z, v4.z);
    adamw_update(c, g4.w, p4.w, m4.w, v4.w);
    reinterpret_cast<float4*>(p)[i] = p4;
    reinterpret_cast<float4*>(m)[i] = m4;
    reinterpret_cast<float4*>(v)[i] = v4;
    if (w) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(p4.x, p4.y), hi = __floats2bfloat162_rn(p4.z, p4.w);
      reinterpret_cast<uint2*>(w)[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    }
  }
  if (blockIdx.x == 0 && threadIdx.x < n - 4 * n4) {
    const int64_t i = 4 * n4 + threadIdx.x;
    float pe = p[i], me = m[i], ve = v[i];
    adamw_update(c, grad[i], pe, me, ve);
    p[i] = pe;
    m[i] = me;
    v[i] = ve;
    if (w) w[i] = __float2bfloat16_rn(pe);
  }
}

// The fused optimizer's step for one vocabulary chunk of a batch of several
// row chunks: part [cols][d] is the chunk's summed dW (chunk-local rows in
// visiting order); row i updates the weights of id v0 + i, or of
// id order[v0 + i] when the vocabulary runs in sorted order. Four weights per
// thread (d is a multiple of 8), adamw_update as everywhere else.
__global__ void __launch_bounds__(256) adamw_rows_kernel(const WsHeader* __restrict__ hdr,
                                                         const float* __restrict__ part, int cols, int d,
                                                         const int32_t* __restrict__ order, int64_t v0,
                                                         float* __restrict__ p, float* __restrict__ m,
                                                         float* __restrict__ v, __nv_bfloat16* __restrict__ w) {
  float c[kAdamwConsts];
  for (int i = 0; i < kAdamwConsts; ++i) c[i] = hdr->opt[i];
  const int q = d / 4;
  const int64_t n4 = (int64_t)cols * q;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const int64_t row = i / q, k = i % q;
    const int64_t id = order ? (int64_t)__ldg(order + v0 + row) : v0 + row;
    const int64_t e = id * q + k;
    const float4 g4 = reinterpret_cast<const float4*>(part)[i];
    float4 p4 = reinterpret_cast<float4*>(p)[e], m4 = reinterpret_cast<float4*>(m)[e],
           v4 = reinterpret_cast<float4*>(v)[e];
    adamw_update(c, g4.x, p4.x, m4.x, v4.x);
    adamw_update(c, g4.y, p4.y, m4.y, v4.y);
    adamw_update(c, g4.z, p4.z, m4.z, v4.z);
    adamw_update(c, g4.w, p4.w, m4.w, v4.w);
    reinterpret_cast<float4*>(p)[e] = p4;
    reinterpret_cast<float4*>(m)[e] = m4;
    reinterpret_cast<float4*>(v)[e] = v4;
    __nv_bfloat162 lo = __floats2bfloat162_rn(p4.x, p4.y), hi = __floats2bfloat162_rn(p4.z, p4.w);
    reinterpret_cast<uint2*>(w)[e] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}

// d(bias) of one staging chunk: out[dst(c)] (=|+=) scale * sum over the
// chunk's rows of G[r][c], with dst(c) = v0 + c, or col_map[v0 + c] when the
// vocabulary runs in sorted order. A block covers 32 columns; thread (c, g)
// sums rows g, g + 8, ... and the 8 partial sums are added in g order.
__global__ void __launch_bounds__(256) dbias_chunk_kernel(const __nv_bfloat16* __restrict__ stage, int ld, int rows,
                                                          int cols, const float* __restrict__ scale,
                                                          float* __restrict__ out, int64_t v0,
                                                          const int32_t* __restrict__ col_map, int accumulate) {
  __shared__ float part[8][32];
  const int c = blockIdx.x * 32 + threadIdx.x, g = threadIdx.y;
  float acc = 0.f;
  if (c < cols)
    for (int r = g; r < rows; r += 8) acc += __bfloat162float(stage[(size_t)r * ld + c]);
  part[g][threadIdx.x] = acc;
  __syncthreads();
  if (g == 0 && c < cols) {
    float t = 0.f;
    for (int k = 0; k < 8; ++k) t += part[k][threadIdx.x];
    t *= __ldg(scale);
    const int64_t dst = col_map ? (int64_t)__ldg(col_map + v0 + c) : v0 + c;
    out[dst] = accumulate ? out[dst] + t : t;
  }
}

// Filter statistics and keep masks of one staging chunk. The chunk's flags
// occupy rows [0, rows) x columns [0, cols) of a row-major array with
// leading dimension ld; a tile whose flag word is zero was filtered out.
// row_keep[r] bit j and col_keep[j] bit r are set when tile (r, j) holds
// gradient (rows <= 64 and cols <= 64 by the workspace plan): the dH and dW
// contractions read one of these words per output tile.
__global__ void count_skipped_kernel(const uint32_t* __restrict__ flags, int rows, int cols, int ld,
                                     WsHeader* hdr, uint64_t* __restrict__ row_keep,
                                     uint64_t* __restrict__ col_keep) {
  __shared__ unsigned red[256];
  unsigned c = 0;
  for (int i = threadIdx.x; i < rows * cols; i += 256) c += flags[(size_t)(i / cols) * ld + (i % cols)] == 0u ? 1u : 0u;
  for (int r = threadIdx.x; r < rows; r += 256) {
    uint64_t k = 0ull;
    for (int j = 0; j < cols; ++j)
      if (flags[(size_t)r * ld + j] != 0u) k |= 1ull << j;
    row_keep[r] = k;
  }
  for (int j = threadIdx.x; j < cols; j += 256) {
    uint64_t k = 0ull;
    for (int r = 0; r < rows; ++r)
      if (flags[(size_t)r * ld + j] != 0u) k |= 1ull << r;
    col_keep[j] = k;
  }
  red[threadIdx.x] = c;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    atomicAdd(&hdr->tiles_total, (unsigned long long)(rows * cols));
    atomicAdd(&hdr->tiles_skipped, (unsigned long long)red[0]);
  }
}

// Ignored-row compaction, one block: idx[i] = original row of the i-th
// valid row (order kept), pos[n] = compact position of row n or -1. Thread t
// owns a contiguous segment of rows; segment counts are scanned in order.
__global__ void __launch_bounds__(1024) compact_index_kernel(const int64_t* __restrict__ y, int64_t n, int64_t vocab,
                                                             int64_t ignore_index, int32_t* __restrict__ idx,
                                                             int32_t* __restrict__ pos) {
  __shared__ int32_t offs[1024];
  const int64_t seg = (n + blockDim.x - 1) / blockDim.x;
  const int64_t r0 = threadIdx.x * seg, r1 = min(n, r0 + seg);
  int32_t c = 0;
  for (int64_t r = r0; r < r1; ++r) {
    const int64_t t = y[r];
    c += (t != ignore_index && t >= 0 && t < vocab) ? 1 : 0;
  }
  offs[threadIdx.x] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t run = 0;
    for (int i = 0; i < (int)blockDim.x; ++i) {
      const int32_t v = offs[i];
      offs[i] = run;
      run += v;
    }
  }
  __syncthreads();
  int32_t o = offs[threadIdx.x];
  for (int64_t r = r0; r < r1; ++r) {
    const int64_t t = y[r];
    if (t != ignore_index && t >= 0 && t < vocab) {
      idx[o] = (int32_t)r;
      pos[r] = o++;
    } else {
      pos[r] = -1;
    }
  }
}

// Row i of the compacted problem: H row, target, LSE and (optional) row
// scale of original row idx[i]. One block per compact row.
__global__ void gather_rows_kernel(const uint4* __restrict__ H, int row_vec, const int32_t* __restrict__ idx,
                                   int64_t count, uint4* __restrict__ Hc, const int64_t* __restrict__ y,
                                   int64_t* __restrict__ yc, const float* __restrict__ lse, float* __restrict__ lsec,
                                   const float* __restrict__ rs, float* __restrict__ rsc) {
  const int64_t i = blockIdx.x;
  if (i >= count) return;
  const int64_t r = idx[i];
  for (int k = threadIdx.x; k < row_vec; k += blockDim.x) Hc[i * row_vec + k] = H[r * row_vec + k];
  if (threadIdx.x == 0) {
    yc[i] = y[r];
    lsec[i] = lse[r];
    if (rs) rsc[i] = rs[r];
  }
}

// dH row n = compacted dH row pos[n], or zeros for an ignored row.
__global__ void scatter_rows_kernel(const float4* __restrict__ dHc, int row_vec, const int32_t* __restrict__ pos,
                                    float4* __restrict__ dH) {
  const int64_t n = blockIdx.x;
  const int32_t p = pos[n];
  for (int k = threadIdx.x; k < row_vec; k += blockDim.x)
    dH[n * row_vec + k] = p >= 0 ? dHc[(int64_t)p * row_vec + k] : make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ host side

// Optional launch timing (flce_profile_set): event pairs around every launch.
struct Profiler {
  std::mutex mu;
  void** events = nullptr;
  int32_t* kinds = nullptr;
  int32_t cap = 0;
  int32_t count = 0;
};
static Profiler g_prof;

struct ProfScope {
  cudaStream_t st;
  int slot = -1;
  ProfScope(int kind, cudaStream_t s) : st(s) {
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (g_prof.events && g_prof.count < g_prof.cap) {
      slot = g_prof.count++;
      g_prof.kinds[slot] = kind;
      cudaEventRecord(static_cast<cudaEvent_t>(g_prof.events[2 * slot]), st);
    }
  }
  ~ProfScope() {
    if (slot >= 0) cudaEventRecord(static_cast<cudaEvent_t>(g_prof.events[2 * slot + 1]), st);
  }
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Plan {
  int64_t n, d, v;
  int nc, vc;            // row chunk; vocabulary chunk the workspace is sized for
  int vcu;               // vocabulary chunk the backward uses (<= vc)
  int n_vtiles;          // ceil(V / 256)
  int row_chunks, v_chunks;
  size_t off_pm, off_ps, off_zy, off_lse, off_bsum, off_flags[2], off_keep[2], off_stage[2];
  size_t off_opt_part;   // fused optimizer, several row chunks: one chunk's dW [Vc][D] fp32 (0 = none)
  // vocabulary sorting (FLCE_FLAG_SORT_VOCAB only)
  size_t off_hpart, off_hmean, off_avg, off_keys[2], off_ids[2], off_inv, off_hist, off_bias_s, off_ys, off_wsort;
  // ignored-row compaction (FLCE_FLAG_COMPACT_IGNORED only)
  size_t off_cidx, off_cpos, off_hc, off_dhc, off_yc, off_lsec, off_rsc;
  size_t total;
};

// Workspace layout for a row chunk of nc rows (a multiple of 256).
static Plan make_plan_rows(const flce_problem& p, int nc) {
  Plan pl{};
  pl.n = p.n_rows;
  pl.d = p.hidden;
  pl.v = p.vocab;
  pl.nc = nc;
  pl.vc = (int)std::min<int64_t>(align_up((size_t)p.vocab, 256), kVocabChunkMax);
  pl.n_vtiles = (int)ceil_div(p.vocab, kBN);
  pl.row_chunks = (int)ceil_div(std::max<int64_t>(p.n_rows, 1), pl.nc);
  pl.vcu = pl.vc;
  pl.v_chunks = (int)ceil_div(p.vocab, pl.vcu);
  size_t off = align_up(sizeof(WsHeader), 1024);
  pl.off_pm = off;
  off = align_up(off + (size_t)pl.n_vtiles * pl.nc * 4, 1024);
  pl.off_ps = off;
  off = align_up(off + (size_t)pl.n_vtiles * pl.nc * 4, 1024);
  pl.off_zy = off;
  off = align_up(off + (size_t)pl.nc * 4, 1024);
  pl.off_lse = off;
  off = align_up(off + (size_t)std::max<int64_t>(p.n_rows, 1) * 4, 1024);
  pl.off_bsum = off;
  off = align_up(off + (size_t)pl.row_chunks * (pl.nc / kCombineRows) * 8, 1024);
  for (int b = 0; b < 2; ++b) {
    pl.off_flags[b] = off;
    off = align_up(off + (size_t)(pl.nc / kBM) * (pl.vc / kBN) * 4, 1024);
    // keep masks: one word per staging row tile, then one per column tile
    pl.off_keep[b] = off;
    off = align_up(off + (size_t)(pl.nc / kBM + pl.vc / kBN) * 8, 1024);
  }
  static_assert(kRowChunk / kBM <= 64 && kVocabChunkMax / kBN <= 64, "a keep mask is one 64-bit word");
  for (int b = 0; b < 2; ++b) {
    pl.off_stage[b] = off;
    off = align_up(off + (size_t)pl.nc * pl.vc * 2, 1024);
  }
  pl.off_opt_part = 0;
  if (pl.row_chunks > 1) {
    pl.off_opt_part = off;
    off = align_up(off + (size_t)pl.vc * p.hidden * 4, 1024);
  }
  if (p.flags & FLCE_FLAG_SORT_VOCAB) {
    // Sizes grow with N and V only, so the plan of a compacted problem (fewer
    // rows, no sort region) ends before this region starts.
    const size_t n = (size_t)std::max<int64_t>(p.n_rows, 1), d = (size_t)p.hidden, v = (size_t)p.vocab;
    pl.off_hpart = off;
    off = align_up(off + (size_t)kHsumMaxSplits * d * 4, 1024);
    pl.off_hmean = off;
    off = align_up(off + d * 4, 1024);
    pl.off_avg = off;
    off = align_up(off + v * 4, 1024);
    for (int b = 0; b < 2; ++b) {
      pl.off_keys[b] = off;
      off = align_up(off + v * 4, 1024);
      pl.off_ids[b] = off;
      off = align_up(off + v * 4, 1024);
    }
    pl.off_inv = off;
    off = align_up(off + v * 4, 1024);
    pl.off_hist = off;
    off = align_up(off + (size_t)256 * ceil_div(p.vocab, kSortTile) * 4, 1024);
    pl.off_bias_s = off;
    off = align_up(off + v * 4, 1024);
    pl.off_ys = off;
    off = align_up(off + n * 8, 1024);
    pl.off_wsort = off;
    off = align_up(off + v * d * 2, 1024);
  }
  if (p.flags & FLCE_FLAG_COMPACT_IGNORED) {
    const size_t n = (size_t)std::max<int64_t>(p.n_rows, 1), d = (size_t)p.hidden;
    pl.off_cidx = off;
    off = align_up(off + n * 4, 1024);
    pl.off_cpos = off;
    off = align_up(off + n * 4, 1024);
    pl.off_hc = off;
    off = align_up(off + n * d * 2, 1024);
    pl.off_dhc = off;
    off = align_up(off + n * d * 4, 1024);
    pl.off_yc = off;
    off = align_up(off + n * 8, 1024);
    pl.off_lsec = off;
    off = align_up(off + n * 4, 1024);
    pl.off_rsc = off;
    off = align_up(off + n * 4, 1024);
  }
  pl.total = off;
  return pl;
}

// Predicted makespan, in 64-deep k-blocks, of the backward launches for a
// vocabulary chunk of vc ids: each launch assigns its tile groups to `slots`
// persistent CTAs (or CTA pairs) round-robin, so a launch lasts as long as its
// busiest slot; `launch_cost` charges each launch's ramp-up and drain.
static double predict_backward(const flce_problem& p, int nc, int vc, int slots, int cluster) {
  const int64_t d_tiles = ceil_div(p.hidden, kBN), kd = ceil_div(p.hidden, kBK);
  const double launch_cost = 24.0;
  std::vector<int64_t> load(slots);
  int64_t next = 0;    // index of the next unit in the current launch
  double total = 0.0;
  auto add = [&](int64_t units, int64_t cost) {
    if (units <= 0) return;
    const int64_t full = units / slots, rem = units % slots;
    for (int c = 0; c < slots; ++c) {
      const int64_t k = (c - next % slots + slots) % slots;   // slot c's position after `next`
      load[c] += (full + (k < rem ? 1 : 0)) * cost;
    }
    next += units;
  };
  auto close = [&]() {
    total += (double)*std::max_element(load.begin(), load.end()) + launch_cost;
    std::fill(load.begin(), load.end(), 0);
    next = 0;
  };
  auto groups = [&](int64_t m_tiles) { return ceil_div(m_tiles, cluster); };
  const int64_t rcs = ceil_div(std::max<int64_t>(p.n_rows, 1), nc), vcs = ceil_div(p.vocab, vc);
  auto dz_units = [&](int64_t s, int64_t& units) {
    const int64_t rows = std::min<int64_t>(nc, p.n_rows - (s / vcs) * nc);
    const int64_t cols = std::min<int64_t>(vc, p.vocab - (s % vcs) * vc);
    units = groups(ceil_div(rows, kBM)) * ceil_div(cols, kBN);
  };
  int64_t u;
  dz_units(0, u);
  add(u, kd);
  close();
  for (int64_t s = 0; s < rcs * vcs; ++s) {
    const int64_t rows = std::min<int64_t>(nc, p.n_rows - (s / vcs) * nc);
    const int64_t cols = std::min<int64_t>(vc, p.vocab - (s % vcs) * vc);
    add(groups(ceil_div(cols, kBM)) * d_tiles, ceil_div(rows, kBK));   // dW
    add(groups(ceil_div(rows, kBM)) * d_tiles, ceil_div(cols, kBK));   // dH
    if (s + 1 < rcs * vcs) {
      dz_units(s + 1, u);
      add(u, kd);
    }
    close();
  }
  return total;
}

// The vocabulary chunk (a multiple of 256, at most the allocated one) with
// the smallest predicted backward makespan; ties go to the larger chunk.
static int choose_vocab_chunk(const flce_problem& p, int nc, int vc_alloc, int slots, int cluster) {
  static std::mutex mu;
  static int64_t key[6] = {-1, -1, -1, -1, -1, -1};
  static int cached = 0;
  std::lock_guard<std::mutex> lock(mu);
  const int64_t k[6] = {p.n_rows, p.hidden, p.vocab, nc, slots, cluster};
  if (std::equal(k, k + 6, key)) return std::min(cached, vc_alloc);
  int best = vc_alloc;
  double best_t = predict_backward(p, nc, vc_alloc, slots, cluster);
  for (int vc = vc_alloc - 256; vc >= std::min(kVocabChunkMin, vc_alloc); vc -= 256) {
    const double t = predict_backward(p, nc, vc, slots, cluster);
    if (t < best_t * 0.9999) {
      best_t = t;
      best = vc;
    }
  }
  std::copy(k, k + 6, key);
  cached = best;
  return best;
}

static Plan make_plan(const flce_problem& p) {
  return make_plan_rows(p, (int)std::min<int64_t>(align_up((size_t)std::max<int64_t>(p.n_rows, 1), 256), kRowChunk));
}

static bool problem_ok(const flce_problem* p) {
  if (!p) return false;
  if (p->n_rows < 0 || p->n_rows > (int64_t)1 << 30) return false;
  if (p->hidden < 1 || p->hidden > (int64_t)1 << 20) return false;
  if (p->vocab < 1 || p->vocab >= (int64_t)1 << 31) return false;
  if (!(p->filter_eps >= 0.f) || !std::isfinite(p->filter_eps)) return false;
  if ((p->flags & ~(FLCE_FLAG_TEST_SHORT_WAITS | FLCE_FLAG_FILTER_FULL_DW | FLCE_FLAG_FILTER_FULL_DH |
                    FLCE_FLAG_COMPACT_IGNORED | FLCE_FLAG_SORT_VOCAB)) != 0u)
    return false;
  return true;
}

static bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D row-major tensor of `outer` rows x `inner` elements, 128-byte swizzle.
static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major operand map (rows of `inner` elements, `outer` rows): when the
// row length is a multiple of 64, a 3-D view (64 elements, rows, inner / 64
// atoms; strides row_bytes and 128 bytes) whose 64 x 64 x 2 box fills both
// swizzle atoms of a 128-wide tile half in one copy; otherwise the 2-D map
// with 64 x 64 boxes. Every address the 3-D view can form lies inside the
// matrix, and rows past `outer` read as zeros as in the 2-D map. Returns the
// layout code the kernels read (kMnBox3d or kMnBoxes2d), 0 on failure.
static int32_t make_map_mn(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return 0;
  if (inner % 64 == 0) {
    cuuint64_t dims[3] = {64, outer, inner / 64};
    cuuint64_t strides[2] = {row_bytes, 128};
    cuuint32_t box[3] = {64, 64, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      return kMnBox3d;
  }
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_bytes, 64, 64) ? kMnBoxes2d : 0;
}

struct DeviceInfo {
  int sms = 0;
  bool ready = false;
};

// Instances of the pair kernel, smallest epilogue set first; a launch takes
// the first whose set holds every problem's mode and whose kSkip matches.
struct PairInstance {
  void (*fn)(const GemmLaunch);
  bool skip;
  int modes;
  uint32_t smem;
};
constexpr int kPairInstances = 5;
static const PairInstance* pair_instances() {
  static const PairInstance inst[kPairInstances] = {
      {flce_gemm_pair_kernel<false, kModesForward>, false, kModesForward, pair_smem_bytes(kModesForward)},
      {flce_gemm_pair_kernel<false, kModesBackward>, false, kModesBackward, pair_smem_bytes(kModesBackward)},
      {flce_gemm_pair_kernel<true, kModesBackward>, true, kModesBackward, pair_smem_bytes(kModesBackward)},
      {flce_gemm_pair_kernel<false, kModesBackwardAdamw>, false, kModesBackwardAdamw,
       pair_smem_bytes(kModesBackwardAdamw)},
      {flce_gemm_pair_kernel<true, kModesBackwardAdamw>, true, kModesBackwardAdamw,
       pair_smem_bytes(kModesBackwardAdamw)},
  };
  return inst;
}

static bool device_setup(int* sms_out) {
  static std::mutex mu;
  static DeviceInfo info[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!info[dev].ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaFuncSetAttribute(flce_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kGemmSmemBytes) != cudaSuccess)
      return false;
    const PairInstance* inst = pair_instances();
    for (int i = 0; i < kPairInstances; ++i)
      if (cudaFuncSetAttribute(inst[i].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)inst[i].smem) !=
          cudaSuccess)
        return false;
    info[dev].sms = sms;
    info[dev].ready = true;
  }
  *sms_out = info[dev].sms;
  return true;
}

// Kernel variant of the GEMM launches:
//   GEMM_CTA1       one CTA per tile, each loading its own A and B;
//   GEMM_PAIR       2-CTA clusters issuing tcgen05.mma.cta_group::2 (M = 256).
// GEMM_PAIR is the default; FLCE_GEMM_MODE=cta1|pair overrides it.
// With filtering, the pair leaves out a k-block only when both of its CTAs
// skip it (coarser dH mask: 256 rows instead of 128).
enum GemmMode { GEMM_CTA1 = 1, GEMM_PAIR = 3 };

static GemmMode gemm_mode() {
  static GemmMode mode = [] {
    const char* e = std::getenv("FLCE_GEMM_MODE");
    if (e && std::strcmp(e, "cta1") == 0) return GEMM_CTA1;
    return GEMM_PAIR;
  }();
  return mode;
}

// Kernel variant of the backward launches, and the vocabulary chunk they use.
static GemmMode backward_mode(const flce_problem&) { return gemm_mode(); }

// The backward groups dW(c), dH(c) and dZ(c+1) into one launch.
// FLCE_BWD_GROUPING=0 launches them one by one instead (for profiling each
// contraction on its own; the same work in more launches).
static bool backward_grouping() {
  static bool on = [] {
    const char* e = std::getenv("FLCE_BWD_GROUPING");
    return !(e && std::strcmp(e, "0") == 0);
  }();
  return on;
}

// FLCE_VOCAB_CHUNK=<ids> (a multiple of 256, for comparisons) overrides the
// model's choice, within the workspace's chunk size.
static int vocab_chunk_override() {
  static const int vc = [] {
    const char* e = std::getenv("FLCE_VOCAB_CHUNK");
    const int v = e ? std::atoi(e) : 0;
    return v >= 256 && v % 256 == 0 ? v : 0;
  }();
  return vc;
}

static void choose_backward_chunk(Plan& pl, const flce_problem& p, int sms) {
  const int cluster = backward_mode(p) == GEMM_CTA1 ? 1 : 2;
  pl.vcu = choose_vocab_chunk(p, pl.nc, pl.vc, std::max(1, sms / cluster), cluster);
  if (vocab_chunk_override()) pl.vcu = std::min(pl.vc, vocab_chunk_override());
  pl.v_chunks = (int)ceil_div(p.vocab, pl.vcu);
}

// Collects up to kMaxProblems GEMM problems for one persistent launch.
struct Group {
  GemmLaunch L;
  int units = 0;
  GemmMode mode;
  int cluster;
  explicit Group(GemmMode m) : mode(m), cluster(m == GEMM_CTA1 ? 1 : 2) { std::memset(&L, 0, sizeof(L)); }
  void add(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& out, const GemmParams& gp) {
    const int u = (int)ceil_div(gp.m_tiles, cluster) * gp.n_tiles;
    if (u <= 0) return;
    const int q = L.n_probs++;
    L.tm_a[q] = a;
    L.tm_b[q] = b;
    L.tm_out[q] = out;
    L.prob[q] = gp;
    units += u;
    L.tile_end[q] = units;
  }
};


// Launches with the fused optimizer can stagger their problems over runs of
// pairs (TileOrder, FLCE_ADAMW_ORDER_GROUPS=k). Measured at the Gravity head
// shape, four runs took 13.84-13.89 ms per step against 13.61 ms in the
// plain order, so the default is the plain order.
static int adamw_order_groups() {
  static const int groups = [] {
    const char* e = std::getenv("FLCE_ADAMW_ORDER_GROUPS");
    const int g = e ? std::atoi(e) : 1;
    return g >= 1 && g <= 64 ? g : 1;
  }();
  return groups;
}

// Programmatic dependent launch of the pair GEMM (FLCE_PDL=0 switches it
// off, for comparisons).
static bool programmatic_launch() {
  static const bool on = [] {
    const char* e = std::getenv("FLCE_PDL");
    return !(e && std::strcmp(e, "0") == 0);
  }();
  return on;
}

static bool launch_group(int kind, const Group& g, int sms, cudaStream_t st) {
  if (g.units <= 0) return true;
  ProfScope prof(kind, st);
  if (g.mode == GEMM_CTA1) {
    const int grid = std::min(g.units, sms);
    flce_gemm_kernel<<<grid, kGemmThreads, kGemmSmemBytes, st>>>(g.L);
    return cudaGetLastError() == cudaSuccess;
  }
  const int grid = 2 * std::min(g.units, sms / 2);
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Programmatic dependent launch: this launch's prologue may overlap the
  // tail of the previous kernel in the stream; the kernel waits for it
  // (griddepcontrol.wait) before touching global memory.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic_launch() ? 2 : 1;
  bool skip = false;
  int modes = 0;
  for (int q = 0; q < g.L.n_probs; ++q) {
    skip = skip || g.L.prob[q].skip_by_flags != 0;
    modes |= 1 << g.L.prob[q].mode;
  }
  const PairInstance* inst = pair_instances();
  for (int i = 0; i < kPairInstances; ++i) {
    if (inst[i].skip != skip || (modes & ~inst[i].modes) != 0) continue;
    cfg.dynamicSmemBytes = inst[i].smem;
    GemmLaunch L = g.L;
    L.order_groups = (modes & kModeAdamw) ? adamw_order_groups() : 1;
    return cudaLaunchKernelEx(&cfg, inst[i].fn, L) == cudaSuccess;
  }
  return false;   // no instance carries this set of epilogues
}

struct Maps {
  CUtensorMap h_k, w_k, w_k_half, h_mn, w_mn, dh, dw;
  CUtensorMap opt_part;   // the fused optimizer's Vc x D dW buffer (several row chunks only)
  CUtensorMap s_store[2], s_k[2], s_mn[2];   // one set per staging buffer
  int32_t h_mn_form = 0, w_mn_form = 0, s_mn_form = 0;   // make_map_mn's layout codes
};

static GemmParams base_params(const flce_problem& p, WsHeader* hdr) {
  GemmParams gp;
  std::memset(&gp, 0, sizeof(gp));
  gp.ignore_index = p.ignore_index;
  gp.status = &hdr->status;
  gp.wait_limit_ns = (p.flags & FLCE_FLAG_TEST_SHORT_WAITS) ? kShortWaitNs : kWaitLimitNs;
  gp.n_rows = (int32_t)p.n_rows;
  gp.n_cols = (int32_t)p.vocab;
  return gp;
}

// prep + forward GEMM + combine per row chunk + finalize.
// reduction: 0 mean, 1 sum, 2 none (per-row losses into loss_rows, `loss` unused).
static flce_status run_forward(const flce_problem& p, const Plan& pl, const Maps& mp, const int64_t* y,
                               float* lse, float* loss, float grad_loss, uint8_t* ws, int sms, cudaStream_t st,
                               const float* bias = nullptr, int reduction = 0, float* loss_rows = nullptr,
                               const int64_t* count_global = nullptr) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  float* part_m = reinterpret_cast<float*>(ws + pl.off_pm);
  float* part_s = reinterpret_cast<float*>(ws + pl.off_ps);
  float* zy = reinterpret_cast<float*>(ws + pl.off_zy);
  double* bsum = reinterpret_cast<double*>(ws + pl.off_bsum);
  {
    ProfScope prof(FLCE_KERNEL_PREP, st);
    prep_kernel<<<1, 1024, 0, st>>>(y, p.n_rows, p.vocab, p.ignore_index, p.filter_eps > 0.f ? 1u : 0u, hdr);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  const int k_blocks = (int)ceil_div(p.hidden, kBK);
  for (int rc = 0; rc < pl.row_chunks && p.n_rows > 0; ++rc) {
    const int64_t r0 = (int64_t)rc * pl.nc;
    const int rows = (int)std::min<int64_t>(pl.nc, p.n_rows - r0);
    GemmParams gp = base_params(p, hdr);
    gp.m_tiles = (int)ceil_div(rows, kBM);
    gp.n_tiles = pl.n_vtiles;
    gp.k_blocks = k_blocks;
    gp.n_fast = 0;
    gp.a_m0 = (int32_t)r0;
    gp.mode = EPI_LSE;
    gp.m_valid = rows;
    gp.row0 = (int32_t)r0;
    gp.col0 = 0;
    gp.part_ld = pl.nc;
    gp.part_t0 = 0;
    gp.y = y;
    gp.part_m = part_m;
    gp.part_s = part_s;
    gp.zy = zy;
    gp.bias = bias;
    const GemmMode gm = gemm_mode();
    Group g(gm);
    g.add(mp.h_k, gm == GEMM_CTA1 ? mp.w_k : mp.w_k_half, mp.h_k, gp);
    if (!launch_group(FLCE_KERNEL_GEMM_LSE, g, sms, st)) return FLCE_ERR_CUDA;
    ProfScope prof(FLCE_KERNEL_COMBINE, st);
    lse_combine_kernel<<<(int)ceil_div(rows, kCombineRows), dim3(kCombineRows, kCombineSplit), 0, st>>>(
        part_m, part_s, pl.nc, pl.n_vtiles, zy, y, r0, rows, p.vocab, p.ignore_index, lse, bsum, loss_rows);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  const int n_blocks = (int)ceil_div(p.n_rows, kCombineRows);
  ProfScope prof(FLCE_KERNEL_FINALIZE, st);
  finalize_kernel<<<1, 256, 0, st>>>(bsum, n_blocks, grad_loss, hdr, loss, reduction, count_global);
  if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  return FLCE_OK;
}

// The backward walks (row chunk, vocabulary chunk) items in order. Item s
// stages its dZ in buffer s % 2. The dZ GEMM of item s+1 shares a launch with
// the dW and dH GEMMs of item s: they touch different staging buffers.
// Fused AdamW on W (flce_forward_backward_adamw): the dW contraction's
// epilogue updates these instead of writing dW.
struct OptTarget {
  float* master;
  float* m;
  float* v;
  __nv_bfloat16* w_out;
};

// vocab_map (sorted vocabulary only): vocabulary position i of this problem
// is id vocab_map[i]; dW rows and d(bias) entries are written to their ids
// in dW_out / dbias, so mp.dw is not used.
static flce_status run_backward(const flce_problem& p, const Plan& pl, const Maps& mp, const int64_t* y,
                                const float* lse, uint8_t* ws, int sms, cudaStream_t st, const float* bias = nullptr,
                                const float* row_scale = nullptr, float* dbias = nullptr,
                                const int32_t* vocab_map = nullptr, float* dW_out = nullptr,
                                const OptTarget* opt = nullptr) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int filter = p.filter_eps > 0.f ? 1 : 0;
  const int d_tiles = (int)ceil_div(p.hidden, kBN);
  const int items = pl.row_chunks * pl.v_chunks;
  // Items run row-chunk-major, except with the fused optimizer over several
  // row chunks: then vocabulary-chunk-major, so that a chunk's dW is complete
  // (summed over the row chunks in a Vc x D buffer) before the next chunk's
  // starts, and its AdamW step runs right after.
  const bool vocab_major = opt && pl.row_chunks > 1;
  auto item_rc_vi = [&](int s, int& rc, int& vi) {
    if (vocab_major) {
      rc = s % pl.row_chunks;
      vi = s / pl.row_chunks;
    } else {
      rc = s / pl.v_chunks;
      vi = s % pl.v_chunks;
    }
  };
  auto item_geom = [&](int s, int64_t& r0, int& rows, int64_t& v0, int& cols) {
    int rc, vi;
    item_rc_vi(s, rc, vi);
    r0 = (int64_t)rc * pl.nc;
    rows = (int)std::min<int64_t>(pl.nc, p.n_rows - r0);
    v0 = (int64_t)vi * pl.vcu;
    cols = (int)std::min<int64_t>(pl.vcu, p.vocab - v0);
  };
  auto dz_params = [&](int s) {
    int64_t r0, v0;
    int rows, cols;
    item_geom(s, r0, rows, v0, cols);
    GemmParams dz = base_params(p, hdr);
    dz.m_tiles = (int)ceil_div(rows, kBM);
    dz.n_tiles = (int)ceil_div(cols, kBN);
    dz.k_blocks = (int)ceil_div(p.hidden, kBK);
    dz.n_fast = 0;
    dz.a_m0 = (int32_t)r0;
    dz.b_n0 = (int32_t)v0;
    dz.mode = EPI_DZ;
    dz.m_valid = rows;
    dz.row0 = (int32_t)r0;
    dz.col0 = (int32_t)v0;
    dz.y = y;
    dz.lse = lse;
    dz.filter = filter;
    dz.filter_eps = p.filter_eps;
    dz.bias = bias;
    dz.row_scale = row_scale;
    dz.flags = reinterpret_cast<uint32_t*>(ws + pl.off_flags[s & 1]);
    dz.flags_ld = pl.vcu / kBN;
    return dz;
  };
  // d(bias) of item s, read from its staging buffer before that buffer is
  // overwritten two items later.
  auto dbias_item = [&](int s) -> bool {
    if (!dbias) return true;
    int64_t r0, v0;
    int rows, cols;
    item_geom(s, r0, rows, v0, cols);
    int rc, vi;
    item_rc_vi(s, rc, vi);
    const __nv_bfloat16* stage = reinterpret_cast<const __nv_bfloat16*>(ws + pl.off_stage[s & 1]);
    ProfScope prof(FLCE_KERNEL_DBIAS, st);
    dbias_chunk_kernel<<<(int)ceil_div(cols, 32), dim3(32, 8), 0, st>>>(stage, pl.vcu, rows, cols, &hdr->scale,
                                                                        dbias, v0, vocab_map, rc > 0 ? 1 : 0);
    return cudaGetLastError() == cudaSuccess;
  };
  // Statistics and keep masks of item s's flags (buffer s % 2), before the
  // contractions of item s read them.
  auto count_skipped = [&](const GemmParams& dz, int s) -> bool {
    if (!filter) return true;
    ProfScope prof(FLCE_KERNEL_FILTER_STATS, st);
    uint64_t* keep = reinterpret_cast<uint64_t*>(ws + pl.off_keep[s & 1]);
    count_skipped_kernel<<<1, 256, 0, st>>>(dz.flags, dz.m_tiles, dz.n_tiles, dz.flags_ld, hdr, keep,
                                            keep + pl.nc / kBM);
    return cudaGetLastError() == cudaSuccess;
  };

  const GemmMode gm = backward_mode(p);
  const CUtensorMap& w_b = gm == GEMM_CTA1 ? mp.w_k : mp.w_k_half;
  {
    Group g(gm);
    const GemmParams dz0 = dz_params(0);
    g.add(mp.h_k, w_b, mp.s_store[0], dz0);
    if (!launch_group(FLCE_KERNEL_GEMM_DZ, g, sms, st)) return FLCE_ERR_CUDA;
    if (!count_skipped(dz0, 0)) return FLCE_ERR_CUDA;
    if (!dbias_item(0)) return FLCE_ERR_CUDA;
  }
  for (int s = 0; s < items; ++s) {
    const int b = s & 1;
    int64_t r0, v0;
    int rows, cols;
    item_geom(s, r0, rows, v0, cols);
    int rc, vi;
    item_rc_vi(s, rc, vi);
    const uint64_t* keep = reinterpret_cast<const uint64_t*>(ws + pl.off_keep[b]);
    Group g(gm);
    // dW[v0 : v0+cols, :] (=|+=) scale * staging^T * H[r0 : r0+rows, :]
    GemmParams dw = base_params(p, hdr);
    dw.m_tiles = (int)ceil_div(cols, kBM);
    dw.n_tiles = d_tiles;
    dw.k_blocks = (int)ceil_div(rows, kBK);
    dw.a_mn = mp.s_mn_form;
    dw.b_mn = mp.h_mn_form;
    dw.n_fast = 1;
    dw.b_k0 = (int32_t)r0;
    dw.mode = rc == 0 ? EPI_STORE : EPI_REDUCE;
    dw.out_m0 = (int32_t)v0;
    dw.scale = &hdr->scale;
    dw.skip_by_flags = filter && !(p.flags & FLCE_FLAG_FILTER_FULL_DW);
    dw.flags_a_is_rows = 0;
    dw.keep = keep + pl.nc / kBM;
    if (vocab_map || opt) {
      dw.m_valid = cols;
      dw.out_rows = vocab_map;
      dw.out_ptr = dW_out;
      dw.out_ld = p.hidden;
      dw.out_cols = (int32_t)p.hidden;
      dw.out_rows_n = (int32_t)p.vocab;
    }
    const CUtensorMap* dw_map = &mp.dw;
    if (opt && !vocab_major) {
      // One row chunk: each dW tile is complete after this contraction.
      dw.mode = EPI_ADAMW;
      dw.out_ptr = opt->master;
      dw.opt = hdr->opt;
      dw.opt_m = opt->m;
      dw.opt_v = opt->v;
      dw.opt_w = opt->w_out;
    } else if (opt) {
      // Several row chunks: the chunk's dW is summed in the Vc x D buffer
      // (chunk-local rows, in the order the vocabulary is visited) and the
      // AdamW step follows the last row chunk (adamw_rows_kernel).
      dw.out_rows = nullptr;
      dw.out_m0 = 0;
      dw_map = &mp.opt_part;
    }
    g.add(mp.s_mn[b], mp.h_mn, *dw_map, dw);
    // dH[r0 : r0+rows, :] (=|+=) scale * staging * W[v0 : v0+cols, :]
    GemmParams dh = base_params(p, hdr);
    dh.m_tiles = (int)ceil_div(rows, kBM);
    dh.n_tiles = d_tiles;
    dh.k_blocks = (int)ceil_div(cols, kBK);
    dh.a_mn = kKMajor;
    dh.b_mn = mp.w_mn_form;
    dh.n_fast = 1;
    dh.b_k0 = (int32_t)v0;
    dh.mode = vi == 0 ? EPI_STORE : EPI_REDUCE;
    dh.out_m0 = (int32_t)r0;
    dh.scale = &hdr->scale;
    dh.skip_by_flags = filter && !(p.flags & FLCE_FLAG_FILTER_FULL_DH);
    dh.flags_a_is_rows = 1;
    dh.keep = keep;
    g.add(mp.s_k[b], mp.w_mn, mp.dh, dh);
    GemmParams dz_next;
    const bool has_next = s + 1 < items;
    if (has_next) dz_next = dz_params(s + 1);
    if (backward_grouping()) {
      if (has_next) g.add(mp.h_k, w_b, mp.s_store[b ^ 1], dz_next);
      if (!launch_group(FLCE_KERNEL_GEMM_BWD, g, sms, st)) return FLCE_ERR_CUDA;
    } else {
      Group gw(gm), gh(gm), gz(gm);
      gw.add(mp.s_mn[b], mp.h_mn, *dw_map, dw);
      gh.add(mp.s_k[b], mp.w_mn, mp.dh, dh);
      if (!launch_group(FLCE_KERNEL_GEMM_DW, gw, sms, st)) return FLCE_ERR_CUDA;
      if (!launch_group(FLCE_KERNEL_GEMM_DH, gh, sms, st)) return FLCE_ERR_CUDA;
      if (has_next) {
        gz.add(mp.h_k, w_b, mp.s_store[b ^ 1], dz_next);
        if (!launch_group(FLCE_KERNEL_GEMM_DZ, gz, sms, st)) return FLCE_ERR_CUDA;
      }
    }
    if (vocab_major && rc == pl.row_chunks - 1) {
      // The chunk's dW is complete: its AdamW step, before the next chunk's
      // first contraction overwrites the buffer.
      const float* part = reinterpret_cast<const float*>(ws + pl.off_opt_part);
      const int64_t n4 = (int64_t)cols * p.hidden / 4;
      const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((int64_t)sms * 8, ceil_div(n4, 256)));
      ProfScope prof(FLCE_KERNEL_ADAMW_STEP, st);
      adamw_rows_kernel<<<blocks, 256, 0, st>>>(hdr, part, cols, (int)p.hidden, vocab_map, v0, opt->master, opt->m,
                                                 opt->v, opt->w_out);
      if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
    }
    if (has_next && !count_skipped(dz_next, s + 1)) return FLCE_ERR_CUDA;
    if (has_next && !dbias_item(s + 1)) return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

// The backward, with ignored rows removed first when the problem asks for it.
static flce_status run_backward_any(const flce_problem& p, const Plan& pl, const Maps& mp, const void* H,
                                    const void* W, const int64_t* y, const float* lse, float* dH, float* dW,
                                    uint8_t* ws, int sms, cudaStream_t st, const float* bias, const float* row_scale,
                                    float* dbias, const OptTarget* opt = nullptr);

static bool build_maps(const flce_problem& p, const Plan& pl, const void* H, const void* W, float* dH, float* dW,
                       uint8_t* ws, bool backward, Maps* mp) {
  const uint64_t D = (uint64_t)p.hidden, N = (uint64_t)std::max<int64_t>(p.n_rows, 1), V = (uint64_t)p.vocab;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (!make_map(&mp->h_k, bf, H, D, N, D * 2, 64, kBM)) return false;
  if (!make_map(&mp->w_k, bf, W, D, V, D * 2, 64, kBN)) return false;
  if (!make_map(&mp->w_k_half, bf, W, D, V, D * 2, 64, kBN / 2)) return false;
  if (!backward) return true;
  if (!(mp->h_mn_form = make_map_mn(&mp->h_mn, H, D, N, D * 2))) return false;
  if (!(mp->w_mn_form = make_map_mn(&mp->w_mn, W, D, V, D * 2))) return false;
  for (int b = 0; b < 2; ++b) {
    void* stage = ws + pl.off_stage[b];
    const uint64_t vc = (uint64_t)pl.vcu, nc = (uint64_t)pl.nc;
    if (!make_map(&mp->s_store[b], bf, stage, vc, nc, vc * 2, 64, 32)) return false;
    if (!make_map(&mp->s_k[b], bf, stage, vc, nc, vc * 2, 64, kBM)) return false;
    const int32_t form = make_map_mn(&mp->s_mn[b], stage, vc, nc, vc * 2);
    if (!form || (b == 1 && form != mp->s_mn_form)) return false;
    mp->s_mn_form = form;
  }
  if (!make_map(&mp->dh, f32, dH, D, N, D * 4, 32, 32)) return false;
  if (dW && !make_map(&mp->dw, f32, dW, D, V, D * 4, 32, 32)) return false;
  if (pl.off_opt_part &&
      !make_map(&mp->opt_part, f32, ws + pl.off_opt_part, D, (uint64_t)pl.vc, D * 4, 32, 32))
    return false;
  return true;
}

// Vocabulary sorting (FLCE_FLAG_SORT_VOCAB, Cut Cross-Entropy Sec. 4.3):
// average logit of every id over the valid rows, their stable descending
// order, W, the bias and the targets rearranged in that order, then the
// backward of the rearranged problem, which writes dW and d(bias) back in id
// order. `sp` is the plan that holds the sort buffers: the caller's full
// plan, also when the rows were compacted into `p` (whose own plan `pl` has
// no sort region and ends before it).
static flce_status run_backward_sorted(const flce_problem& p, const Plan& pl, const Plan& sp, const Maps& mp,
                                       const void* H, const void* W, const int64_t* y, const float* lse, float* dW,
                                       uint8_t* ws, int sms, cudaStream_t st, const float* bias,
                                       const float* row_scale, float* dbias, const OptTarget* opt) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int d = (int)p.hidden;
  const int64_t n = p.n_rows, v = p.vocab;
  float* hpart = reinterpret_cast<float*>(ws + sp.off_hpart);
  float* hmean = reinterpret_cast<float*>(ws + sp.off_hmean);
  float* avg = reinterpret_cast<float*>(ws + sp.off_avg);
  uint32_t* keys0 = reinterpret_cast<uint32_t*>(ws + sp.off_keys[0]);
  uint32_t* keys1 = reinterpret_cast<uint32_t*>(ws + sp.off_keys[1]);
  int32_t* order = reinterpret_cast<int32_t*>(ws + sp.off_ids[0]);
  int32_t* ids1 = reinterpret_cast<int32_t*>(ws + sp.off_ids[1]);
  int32_t* inv = reinterpret_cast<int32_t*>(ws + sp.off_inv);
  float* bias_s = bias ? reinterpret_cast<float*>(ws + sp.off_bias_s) : nullptr;
  int64_t* ys = reinterpret_cast<int64_t*>(ws + sp.off_ys);
  void* w_sorted = ws + sp.off_wsort;
  const int splits = hsum_splits(n);
  const unsigned vocab_blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((int64_t)sms * 8, ceil_div(v, 8)));
  {
    ProfScope prof(FLCE_KERNEL_VOCAB_KEYS, st);
    hsum_partial_kernel<<<dim3((unsigned)ceil_div(d, kHsumCols), (unsigned)splits), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(H), n, d, y, v, p.ignore_index, splits, hpart);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  {
    ProfScope prof(FLCE_KERNEL_VOCAB_KEYS, st);
    hmean_kernel<<<(unsigned)ceil_div(d, 256), 256, 0, st>>>(hpart, splits, d, &hdr->count, hmean);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  {
    ProfScope prof(FLCE_KERNEL_VOCAB_KEYS, st);
    avg_logit_kernel<<<vocab_blocks, kVocabWarpsPerBlock * 32, 0, st>>>(static_cast<const __nv_bfloat16*>(W), v, d,
                                                                        hmean, bias, avg, keys0);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  {
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws + sp.off_hist);
    const unsigned tiles = (unsigned)ceil_div(v, kSortTile);
    uint32_t* keys[2] = {keys0, keys1};
    int32_t* ids[2] = {order, ids1};
    for (int pass = 0; pass < 4; ++pass) {
      const int src = pass & 1, shift = 8 * pass;
      {
        ProfScope prof(FLCE_KERNEL_VOCAB_SORT, st);
        radix_hist_kernel<<<tiles, 256, 0, st>>>(keys[src], (int)v, shift, hist);
      }
      {
        ProfScope prof(FLCE_KERNEL_VOCAB_SORT, st);
        radix_scan_kernel<<<1, 1024, 0, st>>>(hist, (int)(256 * tiles));
      }
      {
        ProfScope prof(FLCE_KERNEL_VOCAB_SORT, st);
        radix_scatter_kernel<<<tiles, 256, 0, st>>>(keys[src], pass == 0 ? nullptr : ids[src], (int)v, shift, hist,
                                                    keys[src ^ 1], ids[src ^ 1]);
      }
      if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
    }
    // Four passes end back in keys0 / order.
    ProfScope prof(FLCE_KERNEL_VOCAB_SORT, st);
    radix_inverse_kernel<<<(unsigned)ceil_div(v, 256), 256, 0, st>>>(order, (int)v, inv);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  {
    ProfScope prof(FLCE_KERNEL_VOCAB_GATHER, st);
    gather_vocab_kernel<<<vocab_blocks, kVocabWarpsPerBlock * 32, 0, st>>>(
        static_cast<const uint4*>(W), d / 8, order, v, static_cast<uint4*>(w_sorted), bias, bias_s);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  {
    ProfScope prof(FLCE_KERNEL_VOCAB_GATHER, st);
    remap_targets_kernel<<<(unsigned)ceil_div(n, 256), 256, 0, st>>>(y, n, v, p.ignore_index, inv, ys);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  Maps ms = mp;
  const uint64_t D = (uint64_t)d, V = (uint64_t)v;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&ms.w_k, bf, w_sorted, D, V, D * 2, 64, kBN)) return FLCE_ERR_CUDA;
  if (!make_map(&ms.w_k_half, bf, w_sorted, D, V, D * 2, 64, kBN / 2)) return FLCE_ERR_CUDA;
  if (!(ms.w_mn_form = make_map_mn(&ms.w_mn, w_sorted, D, V, D * 2))) return FLCE_ERR_CUDA;
  // Ignored rows carry target -1 in the sorted problem: a valid sorted
  // position can equal the caller's ignore index when that lies in [0, V).
  flce_problem ps = p;
  ps.ignore_index = -1;
  return run_backward(ps, pl, ms, ys, lse, ws, sms, st, bias_s, row_scale, dbias, order, dW, opt);
}

static flce_status run_backward_any(const flce_problem& p, const Plan& pl, const Maps& mp, const void* H,
                                    const void* W, const int64_t* y, const float* lse, float* dH, float* dW,
                                    uint8_t* ws, int sms, cudaStream_t st, const float* bias, const float* row_scale,
                                    float* dbias, const OptTarget* opt) {
  const bool sorted = (p.flags & FLCE_FLAG_SORT_VOCAB) != 0u;
  auto plain = [&]() {
    return sorted ? run_backward_sorted(p, pl, pl, mp, H, W, y, lse, dW, ws, sms, st, bias, row_scale, dbias, opt)
                  : run_backward(p, pl, mp, y, lse, ws, sms, st, bias, row_scale, dbias, nullptr, nullptr, opt);
  };
  if (!(p.flags & FLCE_FLAG_COMPACT_IGNORED)) return plain();
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  int32_t* idx = reinterpret_cast<int32_t*>(ws + pl.off_cidx);
  int32_t* pos = reinterpret_cast<int32_t*>(ws + pl.off_cpos);
  compact_index_kernel<<<1, 1024, 0, st>>>(y, p.n_rows, p.vocab, p.ignore_index, idx, pos);
  if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  // The valid count sizes every launch below: read it back (one synchronisation).
  int64_t count = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FLCE_ERR_CUDA;
  if (cudaMemcpy(&count, &hdr->count, sizeof(count), cudaMemcpyDeviceToHost) != cudaSuccess) return FLCE_ERR_CUDA;
  // With no valid row the fused optimizer still takes its step (a zero
  // gradient); the uncompacted backward gives it one.
  if (count == p.n_rows || (count == 0 && opt)) return plain();
  if (count == 0) {
    if (cudaMemsetAsync(dH, 0, (size_t)p.n_rows * p.hidden * 4, st) != cudaSuccess) return FLCE_ERR_CUDA;
    if (cudaMemsetAsync(dW, 0, (size_t)p.vocab * p.hidden * 4, st) != cudaSuccess) return FLCE_ERR_CUDA;
    if (dbias && cudaMemsetAsync(dbias, 0, (size_t)p.vocab * 4, st) != cudaSuccess) return FLCE_ERR_CUDA;
    return FLCE_OK;
  }
  void* Hc = ws + pl.off_hc;
  float* dHc = reinterpret_cast<float*>(ws + pl.off_dhc);
  int64_t* yc = reinterpret_cast<int64_t*>(ws + pl.off_yc);
  float* lsec = reinterpret_cast<float*>(ws + pl.off_lsec);
  float* rsc = row_scale ? reinterpret_cast<float*>(ws + pl.off_rsc) : nullptr;
  gather_rows_kernel<<<(unsigned)count, 256, 0, st>>>(static_cast<const uint4*>(H), (int)(p.hidden / 8), idx, count,
                                                      static_cast<uint4*>(Hc), y, yc, lse, lsec, row_scale, rsc);
  if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  flce_problem pc = p;
  pc.n_rows = count;
  pc.flags &= ~(FLCE_FLAG_COMPACT_IGNORED | FLCE_FLAG_SORT_VOCAB);
  // Fits in front of the sort and compaction buffers of the full plan.
  Plan plc = make_plan(pc);
  choose_backward_chunk(plc, pc, sms);
  Maps mpc;
  if (!build_maps(pc, plc, Hc, W, dHc, dW, ws, true, &mpc)) return FLCE_ERR_CUDA;
  flce_status r = sorted ? run_backward_sorted(pc, plc, pl, mpc, Hc, W, yc, lsec, dW, ws, sms, st, bias, rsc, dbias,
                                               opt)
                         : run_backward(pc, plc, mpc, yc, lsec, ws, sms, st, bias, rsc, dbias, nullptr, nullptr, opt);
  if (r != FLCE_OK) return r;
  scatter_rows_kernel<<<(unsigned)p.n_rows, 256, 0, st>>>(reinterpret_cast<const float4*>(dHc), (int)(p.hidden / 4),
                                                          pos, reinterpret_cast<float4*>(dH));
  return cudaGetLastError() == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
}

// forward_only: the call needs only the buffers in front of the backward's
// flags and staging chunks (flce_forward_workspace_bytes).
static flce_status check_common(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                const float* loss, const void* ws, size_t ws_bytes, bool forward_only = false) {
  if (!problem_ok(p)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!loss || !ws) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->n_rows > 0 && (!H || !y)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!W) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(ws, 256)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(y, 8)) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->hidden % 8 != 0) return FLCE_ERR_UNSUPPORTED;
  if (!aligned(H, 16) || !aligned(W, 16)) return FLCE_ERR_UNSUPPORTED;
  const Plan pl = make_plan(*p);
  if (ws_bytes < (forward_only ? pl.off_flags[0] : pl.total)) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  return FLCE_OK;
}

// ------------------------------------------------------------------ static scratch
// Workspace of flce_forward_static_scratch: a fixed array in device memory
// that every GPU loading this library holds until the process exits. Host
// code must not pass the symbol itself to a kernel (on the host it names a
// stand-in object, not device memory); the device address comes from
// cudaGetSymbolAddress, looked up once per device and context: a context
// torn down and created again (cudaDeviceReset) loads the module afresh, and
// the array may then sit at another address.
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

static PFN_cuCtxGetCurrent_v4000 ctx_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

// Called after device_setup, so the device's primary context is current.
static bool static_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  static CUcontext ctx_of[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  CUcontext ctx = nullptr;
  PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_current_fn();
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || ctx_of[dev] != ctx) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_static_scratch) != cudaSuccess || !a) return false;
    addr[dev] = a;
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return true;
}

// Largest row chunk (a multiple of 256, at most the usual one) whose forward
// buffers fit in the static scratch; 0 when even 256 rows do not fit.
static int static_scratch_row_chunk(const flce_problem& p) {
  int nc = (int)std::min<int64_t>(align_up((size_t)std::max<int64_t>(p.n_rows, 1), 256), kRowChunk);
  for (; nc >= 256; nc -= 256)
    if (make_plan_rows(p, nc).off_flags[0] <= kStaticScratchBytes) return nc;
  return 0;
}

}  // namespace flce

using namespace flce;

extern "C" {

size_t flce_workspace_bytes(const flce_problem* p) {
  if (!problem_ok(p)) return 0;
  return make_plan(*p).total;
}

size_t flce_forward_workspace_bytes(const flce_problem* p) {
  if (!problem_ok(p)) return 0;
  return make_plan(*p).off_flags[0];
}

const char* flce_status_string(flce_status s) {
  switch (s) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARGUMENT: return "FLCE_ERR_INVALID_ARGUMENT";
    case FLCE_ERR_WORKSPACE_TOO_SMALL: return "FLCE_ERR_WORKSPACE_TOO_SMALL";
    case FLCE_ERR_BAD_TARGET: return "FLCE_ERR_BAD_TARGET";
    case FLCE_ERR_UNSUPPORTED: return "FLCE_ERR_UNSUPPORTED";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT";
  }
  return "FLCE_UNKNOWN_STATUS";
}

flce_status flce_forward(const flce_problem* p, const void* H, const void* W, const int64_t* y, float* lse,
                         float* loss, void* ws, size_t ws_bytes, void* stream) {
  flce_status s = check_common(p, H, W, y, loss, ws, ws_bytes, true);
  if (s != FLCE_OK) return s;
  if (p->n_rows > 0 && !lse) return FLCE_ERR_INVALID_ARGUMENT;
  int sms = 0;
  if (!device_setup(&sms)) return FLCE_ERR_CUDA;
  const Plan pl = make_plan(*p);
  Maps mp;
  if (p->n_rows > 0 && !build_maps(*p, pl, H, W, nullptr, nullptr, static_cast<uint8_t*>(ws), false, &mp))
    return FLCE_ERR_CUDA;
  return run_forward(*p, pl, mp, y, lse, loss, 1.0f, static_cast<uint8_t*>(ws), sms,
                     static_cast<cudaStream_t>(stream));
}

// flce_forward_backward, and flce_forward_backward_global when count_global
// is not NULL.
static flce_status forward_backward_impl(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                         const int64_t* count_global, float grad_loss, float* lse, float* loss,
                                         float* dH, float* dW, void* ws, size_t ws_bytes, void* stream) {
  flce_status s = check_common(p, H, W, y, loss, ws, ws_bytes);
  if (s != FLCE_OK) return s;
  if (!dW || (p->n_rows > 0 && !dH)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(grad_loss)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(dW, 16) || !aligned(dH, 16)) return FLCE_ERR_UNSUPPORTED;
  int sms = 0;
  if (!device_setup(&sms)) return FLCE_ERR_CUDA;
  Plan pl = make_plan(*p);
  choose_backward_chunk(pl, *p, sms);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* lse_buf = lse ? lse : reinterpret_cast<float*>(wsb + pl.off_lse);
  if (p->n_rows == 0) {
    // No rows: loss 0 and dW = 0.
    Maps none;
    flce_status r = run_forward(*p, pl, none, y, lse_buf, loss, grad_loss, wsb, sms, st, nullptr, 0, nullptr,
                                count_global);
    if (r != FLCE_OK) return r;
    if (cudaMemsetAsync(dW, 0, (size_t)p->vocab * p->hidden * 4, st) != cudaSuccess) return FLCE_ERR_CUDA;
    return FLCE_OK;
  }
  Maps mp;
  if (!build_maps(*p, pl, H, W, dH, dW, wsb, true, &mp)) return FLCE_ERR_CUDA;
  flce_status r = run_forward(*p, pl, mp, y, lse_buf, loss, grad_loss, wsb, sms, st, nullptr, 0, nullptr,
                              count_global);
  if (r != FLCE_OK) return r;
  return run_backward_any(*p, pl, mp, H, W, y, lse_buf, dH, dW, wsb, sms, st, nullptr, nullptr, nullptr);
}

flce_status flce_forward_backward(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                  float grad_loss, float* lse, float* loss, float* dH, float* dW, void* ws,
                                  size_t ws_bytes, void* stream) {
  return forward_backward_impl(p, H, W, y, nullptr, grad_loss, lse, loss, dH, dW, ws, ws_bytes, stream);
}

flce_status flce_count_valid(const flce_problem* p, const int64_t* y, int64_t* count, void* stream) {
  if (!problem_ok(p) || !count || (p->n_rows > 0 && !y)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(y, 8) || !aligned(count, 8)) return FLCE_ERR_INVALID_ARGUMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope prof(FLCE_KERNEL_COUNT, st);
  count_valid_kernel<<<1, 1024, 0, st>>>(y, p->n_rows, p->vocab, p->ignore_index, count);
  return cudaGetLastError() == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
}

flce_status flce_forward_backward_global(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                         const int64_t* count_global, float grad_loss, float* lse, float* loss,
                                         float* dH, float* dW, void* ws, size_t ws_bytes, void* stream) {
  if (!count_global || !aligned(count_global, 8)) return FLCE_ERR_INVALID_ARGUMENT;
  return forward_backward_impl(p, H, W, y, count_global, grad_loss, lse, loss, dH, dW, ws, ws_bytes, stream);
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

flce_status flce_forward_backward_adamw(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                        float grad_loss, float* lse, float* loss, float* dH, float* w_master,
                                        float* adam_m, float* adam_v, void* w_out, const flce_adamw_hparams* hp,
                                        void* ws, size_t ws_bytes, void* stream) {
  flce_status s = check_common(p, H, W, y, loss, ws, ws_bytes);
  if (s != FLCE_OK) return s;
  if (!dH || !w_master || !adam_m || !adam_v || !w_out || !hp) return FLCE_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(grad_loss)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(hp, 8)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(dH, 16) || !aligned(w_master, 16) || !aligned(adam_m, 16) || !aligned(adam_v, 16) ||
      !aligned(w_out, 16))
    return FLCE_ERR_UNSUPPORTED;
  if (p->n_rows < 1) return FLCE_ERR_UNSUPPORTED;
  const size_t wbytes = (size_t)p->vocab * p->hidden * 2;
  if (overlaps(w_out, wbytes, W, wbytes)) return FLCE_ERR_INVALID_ARGUMENT;
  int sms = 0;
  if (!device_setup(&sms)) return FLCE_ERR_CUDA;
  Plan pl = make_plan(*p);
  choose_backward_chunk(pl, *p, sms);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* lse_buf = lse ? lse : reinterpret_cast<float*>(wsb + pl.off_lse);
  Maps mp;
  if (!build_maps(*p, pl, H, W, dH, nullptr, wsb, true, &mp)) return FLCE_ERR_CUDA;
  flce_status r = run_forward(*p, pl, mp, y, lse_buf, loss, grad_loss, wsb, sms, st);
  if (r != FLCE_OK) return r;
  {
    ProfScope prof(FLCE_KERNEL_ADAMW_PREP, st);
    adamw_prep_kernel<<<1, 32, 0, st>>>(hp, reinterpret_cast<WsHeader*>(wsb));
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  const OptTarget opt{w_master, adam_m, adam_v, static_cast<__nv_bfloat16*>(w_out)};
  return run_backward_any(*p, pl, mp, H, W, y, lse_buf, dH, nullptr, wsb, sms, st, nullptr, nullptr, nullptr, &opt);
}

flce_status flce_adamw_step(const flce_adamw_hparams* hp, const float* grad, float* w_master, float* adam_m,
                            float* adam_v, void* w_out, int64_t n, void* ws, void* stream) {
  if (!hp || !grad || !w_master || !adam_m || !adam_v || !ws || n < 0) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(hp, 8) || !aligned(ws, 256)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(grad, 16) || !aligned(w_master, 16) || !aligned(adam_m, 16) || !aligned(adam_v, 16) ||
      (w_out && !aligned(w_out, 8)))
    return FLCE_ERR_UNSUPPORTED;
  int sms = 0;
  if (!device_setup(&sms)) return FLCE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  {
    ProfScope prof(FLCE_KERNEL_ADAMW_PREP, st);
    adamw_prep_kernel<<<1, 32, 0, st>>>(hp, hdr);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  if (n == 0) return FLCE_OK;
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((int64_t)sms * 8, ceil_div(n / 4, 256)));
  ProfScope prof(FLCE_KERNEL_ADAMW_STEP, st);
  adamw_step_kernel<<<(unsigned)blocks, 256, 0, st>>>(hdr, grad, w_master, adam_m, adam_v,
                                                     static_cast<__nv_bfloat16*>(w_out), n);
  return cudaGetLastError() == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
}

flce_status flce_forward_ex(const flce_problem* p, int32_t reduction, const void* H, const void* W, const float* bias,
                            const int64_t* y, float* lse, float* loss, void* ws, size_t ws_bytes, void* stream) {
  flce_status s = check_common(p, H, W, y, loss, ws, ws_bytes, true);
  if (s != FLCE_OK) return s;
  if (reduction < FLCE_REDUCTION_MEAN || reduction > FLCE_REDUCTION_NONE) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->n_rows > 0 && !lse) return FLCE_ERR_INVALID_ARGUMENT;
  int sms = 0;
  if (!device_setup(&sms)) return FLCE_ERR_CUDA;
  const Plan pl = make_plan(*p);
  Maps mp;
  if (p->n_rows > 0 && !build_maps(*p, pl, H, W, nullptr, nullptr, static_cast<uint8_t*>(ws), false, &mp))
    return FLCE_ERR_CUDA;
  return run_forward(*p, pl, mp, y, lse, loss, 1.0f, static_cast<uint8_t*>(ws), sms,
                     static_cast<cudaStream_t>(stream), bias, reduction,
                     reduction == FLCE_REDUCTION_NONE ? loss : nullptr);
}

flce_status flce_backward_ex(const flce_problem* p, int32_t reduction, const void* H, const void* W,
                             const float* bias, const int64_t* y, const float* lse, const float* grad, float* dH,
                             float* dW, float* dbias, void* ws, size_t ws_bytes, void* stream) {
  if (!grad) return FLCE_ERR_INVALID_ARGUMENT;
  flce_status s = check_common(p, H, W, y, grad, ws, ws_bytes);
  if (s != FLCE_OK) return s;
  if (reduction < FLCE_REDUCTION_MEAN || reduction > FLCE_REDUCTION_NONE) return FLCE_ERR_INVALID_ARGUMENT;
  if (!dW || (p->n_rows > 0 && (!dH || !lse))) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(dW, 16) || !aligned(dH, 16)) return FLCE_ERR_UNSUPPORTED;
  int sms = 0;
  if (!device_setup(&sms)) return FLCE_ERR_CUDA;
  Plan pl = make_plan(*p);
  choose_backward_chunk(pl, *p, sms);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(wsb);
  {
    ProfScope prof(FLCE_KERNEL_PREP, st);
    prep_kernel<<<1, 1024, 0, st>>>(y, p->n_rows, p->vocab, p->ignore_index, p->filter_eps > 0.f ? 1u : 0u, hdr);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  {
    ProfScope prof(FLCE_KERNEL_SET_SCALE, st);
    set_scale_kernel<<<1, 32, 0, st>>>(grad, reduction, hdr);
    if (cudaGetLastError() != cudaSuccess) return FLCE_ERR_CUDA;
  }
  if (p->n_rows == 0) {
    if (cudaMemsetAsync(dW, 0, (size_t)p->vocab * p->hidden * 4, st) != cudaSuccess) return FLCE_ERR_CUDA;
    if (dbias && cudaMemsetAsync(dbias, 0, (size_t)p->vocab * 4, st) != cudaSuccess) return FLCE_ERR_CUDA;
    return FLCE_OK;
  }
  Maps mp;
  if (!build_maps(*p, pl, H, W, dH, dW, wsb, true, &mp)) return FLCE_ERR_CUDA;
  return run_backward_any(*p, pl, mp, H, W, y, lse, dH, dW, wsb, sms, st, bias,
                          reduction == FLCE_REDUCTION_NONE ? grad : nullptr, dbias);
}

flce_status flce_get_vocab_order(const flce_problem* p, const void* ws, int32_t* order, float* avg_logit,
                                 void* stream) {
  if (!problem_ok(p) || !(p->flags & FLCE_FLAG_SORT_VOCAB)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!ws || !aligned(ws, 256) || !order || !aligned(order, 4)) return FLCE_ERR_INVALID_ARGUMENT;
  if (avg_logit && !aligned(avg_logit, 4)) return FLCE_ERR_INVALID_ARGUMENT;
  const Plan pl = make_plan(*p);
  const uint8_t* wsb = static_cast<const uint8_t*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)p->vocab * 4;
  if (cudaMemcpyAsync(order, wsb + pl.off_ids[0], bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (avg_logit &&
      cudaMemcpyAsync(avg_logit, wsb + pl.off_avg, bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}

flce_status flce_get_device_status(void* ws, void* stream) {
  if (!ws || !aligned(ws, 256)) return FLCE_ERR_INVALID_ARGUMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t status = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FLCE_ERR_CUDA;
  if (cudaMemcpy(&status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return FLCE_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpy(ws, &zero, sizeof(uint32_t), cudaMemcpyHostToDevice) != cudaSuccess) return FLCE_ERR_CUDA;
  if (status & kDevTimeout) return FLCE_ERR_TIMEOUT;
  if (status & kDevBadHparams) return FLCE_ERR_INVALID_ARGUMENT;
  if (status & kDevBadTarget) return FLCE_ERR_BAD_TARGET;
  return FLCE_OK;
}

flce_status flce_get_filter_stats(void* ws, void* stream, double* skipped_fraction) {
  if (!ws || !skipped_fraction || !aligned(ws, 256)) return FLCE_ERR_INVALID_ARGUMENT;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FLCE_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, ws, sizeof(WsHeader), cudaMemcpyDeviceToHost) != cudaSuccess) return FLCE_ERR_CUDA;
  *skipped_fraction = (h.filter_on && h.tiles_total) ? (double)h.tiles_skipped / (double)h.tiles_total : 0.0;
  return FLCE_OK;
}

flce_status flce_forward_static_scratch(const flce_problem* p, const void* H, const void* W, const int64_t* y,
                                        float* lse, float* loss, void* stream) {
  if (!problem_ok(p) || !loss || !W || (p->n_rows > 0 && (!H || !y || !lse))) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(y, 8)) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->hidden % 8 != 0 || !aligned(H, 16) || !aligned(W, 16)) return FLCE_ERR_UNSUPPORTED;
  const int nc = static_scratch_row_chunk(*p);
  if (nc == 0) return FLCE_ERR_UNSUPPORTED;   // the problem's buffers exceed the static scratch
  int sms = 0;
  if (!device_setup(&sms)) return FLCE_ERR_CUDA;
  void* scratch = nullptr;
  if (!static_scratch_address(&scratch)) return FLCE_ERR_CUDA;
  const Plan pl = make_plan_rows(*p, nc);
  Maps mp;
  if (p->n_rows > 0 && !build_maps(*p, pl, H, W, nullptr, nullptr, static_cast<uint8_t*>(scratch), false, &mp))
    return FLCE_ERR_CUDA;
  return run_forward(*p, pl, mp, y, lse, loss, 1.0f, static_cast<uint8_t*>(scratch), sms,
                     static_cast<cudaStream_t>(stream));
}

flce_status flce_profile_set(void** events, int32_t* kinds, int32_t cap) {
  if (cap < 0 || (cap > 0 && (!events || !kinds))) return FLCE_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.events = cap > 0 ? events : nullptr;
  g_prof.kinds = cap > 0 ? kinds : nullptr;
  g_prof.cap = cap;
  g_prof.count = 0;
  return FLCE_OK;
}

int32_t flce_profile_count(void) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  return g_prof.count;
}

}  // extern "C"
