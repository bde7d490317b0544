// Persistent, warp-specialised tcgen05 GEMM with the fused epilogues of the
// LM-head cross-entropy.
//
// One CTA per SM, 192 threads:
//   warp 0      TMA producer: streams 128x64 A and 256x64 B bf16 tiles
//               (128-byte swizzle) into a 4-stage shared-memory ring;
//   warp 1      MMA issuer: one lane issues tcgen05.mma (M=128, N=256, K=16)
//               into one of two 256-column fp32 TMEM accumulators;
//   warps 2..5  epilogue: tcgen05.ld the 128x256 accumulator (one thread per
//               row) and apply one of five epilogues:
//     EPI_LSE    per-row max and sum of exp over the tile's 256 vocabulary
//                columns, written as one (max, sum) partial per row and tile,
//                plus the target logit when the row's target falls in the
//                tile (the blockwise log-sum-exp of Cut Cross-Entropy,
//                Sec. 4.2 Alg. 2, fused with the indexed matmul of Alg. 1);
//     EPI_DZ     G = exp(z - LSE) - onehot(y) for valid rows, 0 otherwise,
//                rounded to bf16 and stored by TMA into a staging chunk
//                (Sec. 4.3 Alg. 4, softmax without renormalisation), with an
//                optional per-tile flag recording whether any |G| >= eps;
//     EPI_STORE  fp32 tile times a device scalar, stored by TMA;
//     EPI_REDUCE fp32 tile times a device scalar, added into global memory
//                by a TMA reduce-add (one writer per element per launch, so
//                the summation order is fixed by the launch order);
//     EPI_ADAMW  fp32 weight-gradient tile times a device scalar, consumed
//                at once by an AdamW update of the weights it belongs to
//                (fp32 master, moments, bf16 copy) and never stored.
// STORE and REDUCE may also write through a row map (plain stores or
// vector reductions instead of TMA) when the rows are in a sorted order.
//
// The accumulator of tile i lives in TMEM buffer i % 2, so the MMA of the next
// tile overlaps the epilogue of the current one. Operands may be K-major or
// MN-major in global memory; both are expressed with 128-byte-swizzled shared
// memory descriptors, so no operand is ever transposed in memory.
#pragma once

#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>

#include "ptx_sm103.cuh"

namespace flce {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;          // 16 KiB
constexpr uint32_t kBBytes = kBN * kBK * 2;          // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;  // 48 KiB
constexpr uint32_t kEpiBoxBytes = 32 * 128;          // 32 rows x 128 bytes
constexpr uint32_t kEpiBytes = 4 * 2 * kEpiBoxBytes; // 4 warps, double buffered
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBarrierBytes = 256;
constexpr uint32_t kGemmSmemBytes = 1024 + kStages * kStageBytes + kEpiBytes + kBarrierBytes;

constexpr float kLog2e = 1.4426950408889634f;

enum EpiMode : int32_t { EPI_LSE = 0, EPI_DZ = 1, EPI_STORE = 2, EPI_REDUCE = 3, EPI_ADAMW = 4 };

// Device constants of one fused AdamW step, in the order the epilogue reads
// them: lr / (1 - beta1^t), 1 / sqrt(1 - beta2^t), 1 - lr * weight_decay,
// beta1, beta2, eps.
constexpr int kAdamwConsts = 6;

// One AdamW update of one weight: c holds the kAdamwConsts step constants
// (lr / (1 - beta1^t), 1 / sqrt(1 - beta2^t), 1 - lr * wd, beta1, beta2,
// eps). Every rounding is spelled out, so the fused epilogue and the
// standalone step give the same bits for the same gradient.
__device__ __forceinline__ void adamw_update(const float* c, float g, float& p, float& m, float& v) {
  m = fmaf(c[3], m, __fmul_rn(__fsub_rn(1.f, c[3]), g));
  v = fmaf(c[4], v, __fmul_rn(__fmul_rn(__fsub_rn(1.f, c[4]), g), g));
  const float q = __fdiv_rn(m, fmaf(sqrtf(v), c[1], c[5]));
  p = fmaf(-c[0], q, __fmul_rn(p, c[2]));
}

// Device status bits (OR-ed into the workspace status word).
constexpr uint32_t kDevBadTarget = 1u;
constexpr uint32_t kDevTimeout = 2u;
constexpr uint32_t kDevBadHparams = 4u;

// How an operand's k-block reaches shared memory. K-major: one box of 64 k
// (128 bytes) by the tile's rows. MN-major (k varies slowest in global
// memory): each 64-element-wide, 128-byte-swizzled atom of the tile is one
// 2-D box of 64 x 64 (kMnBoxes2d), or the map views the rows as (64
// elements, k, atoms) and one 3-D box brings two neighbouring atoms
// (kMnBox3d). The 3-D view needs the row length to be a multiple of 64;
// measured at the Gravity head shape it took the dW and dH k-blocks from
// 560-565 to 530-537 cycles, with bit-identical results.
constexpr int32_t kKMajor = 0, kMnBoxes2d = 1, kMnBox3d = 2;

// Each problem's parameters start on a 128-byte boundary of the launch's
// parameter block. Measured on GB300 with the same sources otherwise: with
// sizes of 224, 264 or 320 bytes (or 64-byte alignment) the forward launch ran
// about 11% slower, at higher SM clocks, than with 128-byte alignment.
struct alignas(128) GemmParams {
  int32_t m_tiles, n_tiles, k_blocks;
  int32_t a_mn, b_mn;          // operand layout: kKMajor, kMnBoxes2d or kMnBox3d
  int32_t n_fast;              // tile raster: 1 = n index varies fastest
  int32_t a_m0, a_k0;          // coordinate offsets of A (M and K directions)
  int32_t b_n0, b_k0;          // coordinate offsets of B (N and K directions)
  int32_t mode;                // EpiMode
  // epilogue geometry
  int32_t m_valid;             // local rows >= m_valid are padding
  int32_t row0;                // global row of local row 0 (LSE / DZ)
  int32_t n_rows;              // N: global rows >= N are padding
  int32_t col0;                // global vocabulary id of local column 0 (LSE / DZ)
  int32_t n_cols;              // V: vocabulary ids >= V are padding (LSE / DZ)
  int32_t out_m0;              // STORE / REDUCE: row coordinate offset in the output map
  int32_t part_ld;             // LSE: leading dimension of the partial arrays
  int32_t part_t0;             // LSE: partial index of n-tile 0
  int32_t filter;              // DZ: write the per-tile skip flags
  int32_t skip_by_flags;       // STORE/REDUCE/ADAMW: leave out k-blocks whose dZ tiles were filtered
  float filter_eps;
  int64_t ignore_index;
  const int64_t* y;
  const float* lse;            // DZ: natural-log LSE per global row
  const float* bias;           // LSE / DZ: optional fp32 bias per vocabulary id (logit = h.w + b)
  const float* row_scale;      // DZ: optional per-global-row factor applied to G before rounding
  float* part_m;               // LSE: running max (log2 units) [tiles][part_ld]
  float* part_s;               // LSE: sum of 2^(t - max)       [tiles][part_ld]
  float* zy;                   // LSE: target logit per local row
  const float* scale;          // STORE / REDUCE: device scalar multiplier
  uint32_t* flags;             // DZ: per staging tile, 4 quarter flags packed in one word
  int32_t flags_ld;            // DZ: staging tiles per staging row-tile
  int32_t flags_a_is_rows;     // skip lookup: 1 = K indexes staging columns (dH), 0 = staging rows (dW)
  const uint64_t* keep;        // skip lookup: the chunk's keep masks (see tile_keep)
  // STORE / REDUCE with a row map: local row r is written to row
  // out_rows[out_m0 + r] of out_ptr (leading dimension out_ld, out_cols
  // columns) by plain stores or vector reductions instead of TMA; rows with
  // out_m0 + r >= out_rows_n or r >= m_valid are padding.
  const int32_t* out_rows;
  float* out_ptr;
  int64_t out_ld;
  int32_t out_cols;
  int32_t out_rows_n;
  // EPI_ADAMW: the tile is the gradient of rows of the fp32 master weights
  // out_ptr; it updates them, the moments opt_m / opt_v (same layout) and
  // writes the bf16 copy opt_w, and the gradient itself is dropped.
  const float* opt;            // kAdamwConsts device values
  float* opt_m;
  float* opt_v;
  __nv_bfloat16* opt_w;
  uint32_t* status;
  uint64_t wait_limit_ns;
};

// One persistent launch runs up to kMaxProblems independent GEMM problems back
// to back: tiles [0, tile_end[0]) belong to problem 0, [tile_end[0],
// tile_end[1]) to problem 1, and so on. Problems in one launch must not read
// what another writes.
constexpr int kMaxProblems = 3;

struct GemmLaunch {
  CUtensorMap tm_a[kMaxProblems];
  CUtensorMap tm_b[kMaxProblems];
  CUtensorMap tm_out[kMaxProblems];
  GemmParams prob[kMaxProblems];
  int32_t n_probs;
  int32_t tile_end[kMaxProblems];
  int32_t order_groups;        // pair kernel: TileOrder groups (1 = plain order)
};
static_assert(sizeof(GemmParams) % 128 == 0 && offsetof(GemmLaunch, prob) % 128 == 0,
              "problem parameters on 128-byte boundaries");
static_assert(sizeof(GemmLaunch) <= 4096, "kernel parameter block");

// Tiles are counted in groups of `cluster` vertically adjacent m-tiles that
// share one n-tile (an SM pair of the pair kernel); with cluster = 1 a group
// is a tile.
__device__ __forceinline__ int m_groups(const GemmParams& p, int cluster) { return (p.m_tiles + cluster - 1) / cluster; }

__device__ __forceinline__ int decode_tile(const GemmLaunch& L, int t, int& pi) {
  pi = 0;
  while (pi < L.n_probs - 1 && t >= L.tile_end[pi]) ++pi;
  return pi == 0 ? t : t - L.tile_end[pi - 1];
}

__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int cluster, int rank, int& mt, int& nt) {
  int mg;
  if (p.n_fast) {
    nt = t % p.n_tiles;
    mg = t / p.n_tiles;
  } else {
    const int groups = m_groups(p, cluster);
    mg = t % groups;
    nt = t / groups;
  }
  mt = mg * cluster + rank;
}

// Which k-blocks of a dW or dH tile read some kept gradient. Before the
// contractions of a staging chunk run, one small kernel turns the chunk's
// per-tile flags (staging tiles are 128 rows x 256 columns) into two bit
// masks, so a tile reads one 64-bit word instead of a flag per k-block:
//   dH (flags_a_is_rows = 1): keep[mt] has bit j set when staging tile
//       (mt, j) holds gradient; k-block kb reads staging columns kb*64..,
//       i.e. unit j = kb*64/256;
//   dW (flags_a_is_rows = 0): keep[c] has bit r set when staging tile (r, c)
//       holds gradient; the tile's vocabulary rows mt*128.. lie in staging
//       column tile c = mt*128/256, and k-block kb reads staging rows
//       kb*64.., i.e. unit r = kb*64/128.
// Bit u of the returned word is set when unit u holds gradient for any of
// the `group` vertically adjacent tiles from mt_first (an SM pair, or a
// cluster, leaves a k-block out only when every one of its tiles does).
__device__ __forceinline__ uint64_t tile_keep(const GemmParams& p, int mt_first, int group) {
  uint64_t k = 0ull;
  for (int r = 0; r < group; ++r) {
    const int mt = mt_first + r;
    if (mt < p.m_tiles) k |= __ldg(p.keep + (p.flags_a_is_rows ? mt : (mt * kBM) / kBN));
  }
  return k;
}

__device__ __forceinline__ bool kblock_dropped(const GemmParams& p, uint64_t keep, int kb) {
  const int unit = p.flags_a_is_rows ? (kb * kBK) / kBN : (kb * kBK) / kBM;
  return ((keep >> unit) & 1ull) == 0ull;
}

__device__ __forceinline__ void record_timeout(uint32_t* status, volatile uint32_t* abort_flag) {
  *abort_flag = 1u;
  atomicOr(status, kDevTimeout);
}

// Epilogue of one accumulator tile, run by the four epilogue warps with one
// tile row per thread (TMEM lane quarter q, lane `lane`). Each warp reports
// through `rel`, once it has read the whole accumulator, that the TMEM buffer
// may be reused; `ebuf` is the warp's staging-box toggle.
struct AccRelease {
  uint64_t* local;          // barrier in this CTA, or
  uint32_t cluster_addr;    // its shared::cluster address in the MMA-issuing CTA
  bool remote;
  bool none = false;        // a tile written without an accumulator: nothing to release
  __device__ __forceinline__ void arrive() const {
    if (none) return;
    if (remote)
      ptx::mbar_arrive_cluster(cluster_addr);
    else
      ptx::mbar_arrive(local);
  }
};

// Epilogue sets a kernel instance is built with: the forward's launches
// need only EPI_LSE, the backward's EPI_DZ, EPI_STORE and EPI_REDUCE, the
// fused optimizer's also EPI_ADAMW. An instance carries only its set's code.
constexpr int kModeLse = 1 << EPI_LSE;
constexpr int kModeDz = 1 << EPI_DZ;
constexpr int kModeStore = (1 << EPI_STORE) | (1 << EPI_REDUCE);
constexpr int kModeAdamw = 1 << EPI_ADAMW;
constexpr int kModesForward = kModeLse;
constexpr int kModesBackward = kModeDz | kModeStore;
constexpr int kModesBackwardAdamw = kModesBackward | kModeAdamw;
constexpr int kModesAll = kModeLse | kModeDz | kModeStore | kModeAdamw;

// `group` CTAs compute each tile group together (1, or 2 for the pair
// kernel); a k-block left out of the MMAs is one every CTA of the group skips.
// A problem whose mode is not in kModes (the host never launches one) only
// releases the accumulator.
template <int kModes = kModesAll>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const CUtensorMap* tmOut, int mt, int nt,
                                              uint32_t taddr, int q, int lane, uint8_t* my_boxes, uint32_t& ebuf,
                                              const AccRelease& rel, int group = 1) {
  const int r_local = q * 32 + lane;
  const int lrow = mt * kBM + r_local;         // local row of this launch
  if (mt >= p.m_tiles) {
    // The empty half of a cluster's last group: nothing to write.
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) rel.arrive();
  } else if ((kModes & kModeLse) && p.mode == EPI_LSE) {
    const bool in_rows = lrow < p.m_valid && (p.row0 + lrow) < p.n_rows;
    const int grow = p.row0 + lrow;
    const int col_t0 = p.col0 + nt * kBN;
    int yl = -1;
    if (in_rows) {
      const int64_t yv = __ldg(p.y + grow);
      if (yv != p.ignore_index && yv >= 0 && yv < p.n_cols) yl = (int)(yv - col_t0);
    }
    const bool ragged = col_t0 + kBN > p.n_cols;
    float run_max = -INFINITY, run_sum = 0.f, zt = 0.f;
    bool has_t = false;
#pragma unroll 1
    for (int c = 0; c < kBN; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(taddr + c, r);
      ptx::tmem_ld_wait();
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
      if (p.bias) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col_t0 + c + j < p.n_cols) x[j] += __ldg(p.bias + col_t0 + c + j);
      }
      if (ragged) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col_t0 + c + j >= p.n_cols) x[j] = -INFINITY;
      }
      if ((unsigned)(yl - c) < 32u) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == yl - c) zt = x[j];
        has_t = true;
      }
      float cmax = x[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, x[j]);
      const float new_max = fmaxf(run_max, cmax * kLog2e);
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) acc += ptx::ex2_approx(fmaf(x[j], kLog2e, -new_max));
      run_sum = run_sum * ptx::ex2_approx(run_max - new_max) + acc;
      run_max = new_max;
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) rel.arrive();
    if (in_rows) {
      const size_t idx = (size_t)(p.part_t0 + nt) * p.part_ld + lrow;
      p.part_m[idx] = run_max;
      p.part_s[idx] = run_sum;
      if (has_t) p.zy[lrow] = zt;
    }
  } else if ((kModes & kModeDz) && p.mode == EPI_DZ) {
    const int grow = p.row0 + lrow;
    const bool in_rows = lrow < p.m_valid && grow < p.n_rows;
    const int col_t0 = p.col0 + nt * kBN;
    bool valid = false;
    int yl = -1;
    float lse2 = 0.f, rs = 1.f;
    if (in_rows) {
      const int64_t yv = __ldg(p.y + grow);
      valid = yv != p.ignore_index && yv >= 0 && yv < p.n_cols;
      if (valid) {
        yl = (int)(yv - col_t0);
        lse2 = __ldg(p.lse + grow) * kLog2e;
        if (p.row_scale) rs = __ldg(p.row_scale + grow);
      }
    }
    const bool ragged = col_t0 + kBN > p.n_cols;
    float amax = 0.f;
#pragma unroll 1
    for (int box = 0; box < kBN / 64; ++box) {
      uint8_t* sbox = my_boxes + ebuf * kEpiBoxBytes;
      if (lane == 0) ptx::bulk_wait_group_read<1>();
      __syncwarp();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int c = box * 64 + half * 32;
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(taddr + c, r);
        ptx::tmem_ld_wait();
        float g[32];
        if (p.bias) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col_t0 + c + j < p.n_cols) r[j] = __float_as_uint(__uint_as_float(r[j]) + __ldg(p.bias + col_t0 + c + j));
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
          g[j] = valid ? ptx::ex2_approx(fmaf(__uint_as_float(r[j]), kLog2e, -lse2)) : 0.f;
        if (ragged) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col_t0 + c + j >= p.n_cols) g[j] = 0.f;
        }
        if ((unsigned)(yl - c) < 32u) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == yl - c) g[j] -= 1.f;
        }
        if (p.filter) {
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(g[j]));
        }
        if (p.row_scale) {
#pragma unroll
          for (int j = 0; j < 32; ++j) g[j] *= rs;
        }
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(g[2 * j], g[2 * j + 1]);
          packed[j] = *reinterpret_cast<uint32_t*>(&b2);
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int chunk = (half * 4 + v) ^ (lane & 7);
          uint4 val = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
          *reinterpret_cast<uint4*>(sbox + lane * 128 + chunk * 16) = val;
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(tmOut, sbox, nt * kBN + box * 64, mt * kBM + q * 32);
        ptx::bulk_commit_group();
      }
      ebuf ^= 1u;
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) rel.arrive();
    if (p.filter) {
      // Staging tile (mt, nt) gets one byte per 32-row quarter; the tile
      // is skipped downstream when the whole 32-bit word is zero.
      const unsigned keep = __any_sync(0xffffffffu, amax >= p.filter_eps) ? 1u : 0u;
      if (lane == 0) reinterpret_cast<uint8_t*>(p.flags + (size_t)mt * p.flags_ld + nt)[q] = (uint8_t)keep;
    }
  } else if ((kModes & (kModeStore | kModeAdamw)) && ((1 << p.mode) & (kModeStore | kModeAdamw))) {
    // EPI_STORE / EPI_REDUCE / EPI_ADAMW
    const bool all_skipped = p.skip_by_flags != 0 && tile_keep(p, mt - mt % group, group) == 0ull;
    const float sc = __ldg(p.scale);
    if ((kModes & kModeAdamw) && p.mode == EPI_ADAMW) {
      // AdamW on the finished gradient tile (the FORGE explainer's fused
      // optimizer), 32 columns at a time. The accumulator gives each thread
      // one row; the slice goes through this warp's shared-memory box so that
      // the weights and moments are read and written row by row instead:
      // lane (rs, j) handles columns 4j..4j+3 of rows rs, rs + 4, ..., rs + 28
      // of the warp's 32, and one warp instruction covers four whole 128-byte
      // lines of each array. (With one row per thread every instruction
      // touched 32 lines, which the small L1 left beside the 230 KiB of
      // shared memory could not hold.) Rows go through out_rows when the
      // vocabulary runs in sorted order. The loads of a slice are issued
      // before the accumulator is read.
      float oc[kAdamwConsts];
#pragma unroll
      for (int i = 0; i < kAdamwConsts; ++i) oc[i] = __ldg(p.opt + i);
      // An earlier tile's TMA stores may still be reading the boxes.
      if (lane == 0) ptx::bulk_wait_group_read<0>();
      __syncwarp();
      const int rs = lane >> 3, jc = lane & 7;
      const int row_base = mt * kBM + q * 32;    // local row of the warp's row 0
      int64_t drow[8];
      bool rok[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int lr = row_base + rs + 4 * k;
        const int sr = p.out_m0 + lr;
        rok[k] = lr < p.m_valid && sr < p.out_rows_n;
        drow[k] = rok[k] ? (p.out_rows ? (int64_t)__ldg(p.out_rows + sr) : (int64_t)sr) * p.out_ld : 0;
      }
#pragma unroll 1
      for (int c = 0; c < kBN; c += 32) {
        const int col = nt * kBN + c + 4 * jc;   // out_cols is a multiple of 8, so 4 columns are all in or out
        const bool col_ok = col < p.out_cols;
        float4 pv[8], mv[8], vv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (rok[k] && col_ok) {
            pv[k] = *reinterpret_cast<const float4*>(p.out_ptr + drow[k] + col);
            mv[k] = *reinterpret_cast<const float4*>(p.opt_m + drow[k] + col);
            vv[k] = *reinterpret_cast<const float4*>(p.opt_v + drow[k] + col);
          }
        }
        uint8_t* sbox = my_boxes + ebuf * kEpiBoxBytes;
        {
          float x[32];
          if (all_skipped) {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = 0.f;
          } else {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(taddr + c, r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) * sc;
          }
          // row `lane`, 16-byte chunk v at chunk v ^ (lane & 7)
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(sbox + lane * 128 + ((v ^ (lane & 7)) * 16)) =
                make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int r = rs + 4 * k;
          const float4 g4 = *reinterpret_cast<const float4*>(sbox + r * 128 + ((jc ^ (r & 7)) * 16));
          if (!(rok[k] && col_ok)) continue;
          float* pe = &pv[k].x;
          float* me = &mv[k].x;
          float* ve = &vv[k].x;
          const float g[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) adamw_update(oc, g[e], pe[e], me[e], ve[e]);
          *reinterpret_cast<float4*>(p.out_ptr + drow[k] + col) = pv[k];
          *reinterpret_cast<float4*>(p.opt_m + drow[k] + col) = mv[k];
          *reinterpret_cast<float4*>(p.opt_v + drow[k] + col) = vv[k];
          __nv_bfloat162 lo = __floats2bfloat162_rn(pe[0], pe[1]), hi = __floats2bfloat162_rn(pe[2], pe[3]);
          *reinterpret_cast<uint2*>(p.opt_w + drow[k] + col) =
              make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        }
        ebuf ^= 1u;                              // the next slice writes the other box
      }
      __syncwarp();
    } else if (p.out_rows) {
      // Row-mapped output (a vocabulary visited in sorted order writes dW
      // rows back in id order; the map is a permutation of the output rows).
      // As in the AdamW epilogue, each 32-column slice goes through the
      // warp's shared-memory box, so that lane (rs, j) writes columns
      // 4j..4j+3 of rows rs, rs + 4, ..., rs + 28 and one instruction covers
      // four whole 128-byte lines.
      if (!(all_skipped && p.mode == EPI_REDUCE)) {
        if (lane == 0) ptx::bulk_wait_group_read<0>();   // earlier TMA stores may still read the boxes
        __syncwarp();
        const int rs = lane >> 3, jc = lane & 7;
        const int row_base = mt * kBM + q * 32;
        int64_t drow[8];
        bool rok[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int lr = row_base + rs + 4 * k;
          const int sr = p.out_m0 + lr;
          rok[k] = lr < p.m_valid && sr < p.out_rows_n;
          drow[k] = rok[k] ? (int64_t)__ldg(p.out_rows + sr) * p.out_ld : 0;
        }
#pragma unroll 1
        for (int c = 0; c < kBN; c += 32) {
          uint8_t* sbox = my_boxes + ebuf * kEpiBoxBytes;
          {
            float x[32];
            if (all_skipped) {
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] = 0.f;
            } else {
              uint32_t r[32];
              ptx::tmem_ld_32x32b_x32(taddr + c, r);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) * sc;
            }
#pragma unroll
            for (int v = 0; v < 8; ++v)
              *reinterpret_cast<float4*>(sbox + lane * 128 + ((v ^ (lane & 7)) * 16)) =
                  make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
          }
          __syncwarp();
          const int col = nt * kBN + c + 4 * jc;
          if (col < p.out_cols) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (!rok[k]) continue;
              const int r = rs + 4 * k;
              const float4 g4 = *reinterpret_cast<const float4*>(sbox + r * 128 + ((jc ^ (r & 7)) * 16));
              float* dst = p.out_ptr + drow[k] + col;
              if (p.mode == EPI_REDUCE)
                ptx::red_add_v4(dst, g4.x, g4.y, g4.z, g4.w);
              else
                *reinterpret_cast<float4*>(dst) = g4;
            }
          }
          ebuf ^= 1u;
        }
        __syncwarp();
      }
    } else if (!(all_skipped && p.mode == EPI_REDUCE)) {
#pragma unroll 1
      for (int c = 0; c < kBN; c += 32) {
        uint8_t* sbox = my_boxes + ebuf * kEpiBoxBytes;
        if (lane == 0) ptx::bulk_wait_group_read<1>();
        __syncwarp();
        float x[32];
        if (all_skipped) {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = 0.f;
        } else {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(taddr + c, r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]) * sc;
        }
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const int chunk = v ^ (lane & 7);
          *reinterpret_cast<float4*>(sbox + lane * 128 + chunk * 16) =
              make_float4(x[4 * v], x[4 * v + 1], x[4 * v + 2], x[4 * v + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int32_t c0 = nt * kBN + c, c1 = p.out_m0 + mt * kBM + q * 32;
          if (p.mode == EPI_REDUCE)
            ptx::tma_reduce_add_2d(tmOut, sbox, c0, c1);
          else
            ptx::tma_store_2d(tmOut, sbox, c0, c1);
          ptx::bulk_commit_group();
        }
        ebuf ^= 1u;
      }
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) rel.arrive();
  } else {
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) rel.arrive();
  }
}

// One CTA per 128x256 tile: every CTA loads its own A and B tiles into a
// 4-stage ring and issues tcgen05.mma.cta_group::1 (M = 128). The pair
// kernel (tile_gemm_pair.cuh) is the default; this one is kept for
// comparison (FLCE_GEMM_MODE=cta1).
__global__ void __launch_bounds__(kGemmThreads, 1) flce_gemm_kernel(const __grid_constant__ GemmLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* epi_smem = smem + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_smem + kEpiBytes);
  uint64_t* full_bar = bars;                   // [kStages]
  uint64_t* empty_bar = bars + kStages;        // [kStages]
  uint64_t* acc_full = bars + 2 * kStages;     // [2]
  uint64_t* acc_empty = bars + 2 * kStages + 2;// [2]
  uint64_t* drain_bar = bars + 2 * kStages + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = L.tile_end[L.n_probs - 1];
  const int unit0 = blockIdx.x;
  const int unit_stride = gridDim.x;
  const uint64_t wait_limit_ns = L.prob[0].wait_limit_ns;
  uint32_t* const status = L.prob[0].status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&acc_full[b], 1);
      ptx::mbar_init(&acc_empty[b], 4);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    ptx::fence_mbarrier_init();
    for (int q = 0; q < L.n_probs; ++q) {
      ptx::prefetch_tmap(&L.tm_a[q]);
      ptx::prefetch_tmap(&L.tm_b[q]);
      ptx::prefetch_tmap(&L.tm_out[q]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int32_t last_parity[kStages];
      for (int s = 0; s < kStages; ++s) last_parity[s] = -1;
      bool ok = true;
      for (int t = unit0; t < num_tiles && ok; t += unit_stride) {
        int pi, mt, nt;
        const int tl = decode_tile(L, t, pi);
        const GemmParams& p = L.prob[pi];
        const CUtensorMap* tmA = &L.tm_a[pi];
        const CUtensorMap* tmB = &L.tm_b[pi];
        tile_coords(p, tl, 1, 0, mt, nt);
        const bool may_skip = p.skip_by_flags != 0;
        const uint64_t keep = may_skip ? tile_keep(p, mt, 1) : ~0ull;
        const int k_blocks = p.k_blocks;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (may_skip && kblock_dropped(p, keep, kb)) continue;
          if (!ptx::mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, wait_limit_ns, abort_flag)) {
            record_timeout(status, abort_flag);
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * kStageBytes;
          uint8_t* sb = sa + kABytes;
          ptx::mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
          const int32_t kc = kb * kBK;
          if (p.a_mn == kMnBox3d) {
            ptx::tma_load_3d(sa, tmA, 0, p.a_k0 + kc, (p.a_m0 + mt * kBM) >> 6, &full_bar[stage]);
          } else if (p.a_mn) {
            for (int h = 0; h < kBM / 64; ++h)
              ptx::tma_load_2d(sa + h * 8192, tmA, p.a_m0 + mt * kBM + h * 64, p.a_k0 + kc, &full_bar[stage]);
          } else {
            ptx::tma_load_2d(sa, tmA, p.a_k0 + kc, p.a_m0 + mt * kBM, &full_bar[stage]);
          }
          if (p.b_mn == kMnBox3d) {
            for (int h = 0; h < kBN / 128; ++h)
              ptx::tma_load_3d(sb + h * 16384, tmB, 0, p.b_k0 + kc, ((p.b_n0 + nt * kBN) >> 6) + 2 * h,
                               &full_bar[stage]);
          } else if (p.b_mn) {
            for (int h = 0; h < kBN / 64; ++h)
              ptx::tma_load_2d(sb + h * 8192, tmB, p.b_n0 + nt * kBN + h * 64, p.b_k0 + kc, &full_bar[stage]);
          } else {
            ptx::tma_load_2d(sb, tmB, p.b_k0 + kc, p.b_n0 + nt * kBN, &full_bar[stage]);
          }
          last_parity[stage] = (int32_t)phase;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Leave no copy in flight into shared memory this CTA is about to give up.
        volatile uint32_t never = 0u;
        for (int s = 0; s < kStages; ++s)
          if (last_parity[s] >= 0) ptx::mbar_wait_bounded(&full_bar[s], (uint32_t)last_parity[s], 100000000ull, &never);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t smem_base = ptx::smem_u32(smem);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int i = 0;
      for (int t = unit0; t < num_tiles && ok; t += unit_stride, ++i) {
        int pi, mt, nt;
        const int tl = decode_tile(L, t, pi);
        const GemmParams& p = L.prob[pi];
        tile_coords(p, tl, 1, 0, mt, nt);
        const uint32_t idesc = ptx::idesc_bf16_f32(kBM, kBN, p.a_mn != 0, p.b_mn != 0);
        const uint32_t buf = i & 1, use = i >> 1;
        if (!ptx::mbar_wait_bounded(&acc_empty[buf], (use & 1u) ^ 1u, wait_limit_ns, abort_flag)) {
          record_timeout(status, abort_flag);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        uint32_t accumulate = 0;
        const bool may_skip = p.skip_by_flags != 0;
        const uint64_t keep = may_skip ? tile_keep(p, mt, 1) : ~0ull;
        const int k_blocks = p.k_blocks;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (may_skip && kblock_dropped(p, keep, kb)) continue;
          if (!ptx::mbar_wait_bounded(&full_bar[stage], phase, wait_limit_ns, abort_flag)) {
            record_timeout(status, abort_flag);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = smem_base + stage * kStageBytes;
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t adesc = p.a_mn ? ptx::smem_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                          : ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024);
            const uint64_t bdesc = p.b_mn ? ptx::smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                          : ptx::smem_desc_sw128(b_addr + k * 32, 16, 1024);
            ptx::mma_bf16_ss(d_tmem, adesc, bdesc, idesc, accumulate);
            accumulate = 1;
          }
          ptx::mma_commit(&empty_bar[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&acc_full[buf]);
      }
      // Every MMA this thread issued has completed once the drain barrier flips.
      ptx::mma_commit(drain_bar);
      volatile uint32_t never = 0u;
      ptx::mbar_wait_bounded(drain_bar, 0u, 100000000ull, &never);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                    // TMEM lane quarter this warp may read
    uint8_t* my_boxes = epi_smem + q * 2 * kEpiBoxBytes;
    uint32_t ebuf = 0;
    int i = 0;
    for (int t = unit0; t < num_tiles; t += unit_stride, ++i) {
      int pi, mt, nt;
      const int tl = decode_tile(L, t, pi);
      const GemmParams& p = L.prob[pi];
      const CUtensorMap* tmOut = &L.tm_out[pi];
      tile_coords(p, tl, 1, 0, mt, nt);
      const uint32_t buf = i & 1, use = i >> 1;
      if (!ptx::mbar_wait_bounded(&acc_full[buf], use & 1u, wait_limit_ns, abort_flag)) {
        record_timeout(status, abort_flag);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + buf * kBN + ((uint32_t)(q * 32) << 16);

      const AccRelease rel{&acc_empty[buf], 0u, false};
      epilogue_tile(p, tmOut, mt, nt, taddr, q, lane, my_boxes, ebuf, rel);
    }
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace flce
