// Fine-grained E4M3 quantisation kernels (sm_103a).
//
//   act_quant_rows  -- 1x128 tiles along K (page 1, Figure 7 (a): per token per
//                      128 channels), row-major codes + [M, K/128] scales.
//   act_quant_cols  -- 128x1 tiles along M with transposed output (page 5,
//                      backward-pass passage: re-quantise into 128x1 tiles).
//   weight_quant    -- 128x128 blocks (page 1, Figure 7 (a)), optional
//                      transposed copy of codes and scales for Dgrad.
//
// Scale rule for every tile/block (page 2, online-amax passage; pages 1-2,
// power-of-2 passage): amax = max|x| floored at 2^-64; s = amax/448 and
// multiplier m = 448/amax by IEEE FP32 division (__fdiv_rn), or in power-of-2
// mode s = 2^ceil(log2(amax/448)) and m = 1/s built from the exponent bits.
// Each element costs one IEEE multiply x*m and one saturating RNE conversion.
// All three kernels are HBM-bound: 16-byte coalesced loads, warp-shuffle amax,
// packed e4m3x2 conversion, and grids sized in multiples of the SM count.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace fp8fg {

namespace {

// 16-byte streaming load (read once; do not keep in L1).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Unpack a 16-byte vector into floats: 8 BF16 or 4 FP32 values.
template <typename T>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

// --------------------------------------------------------------------------
// 1x128 tiles along K.  With K % 128 == 0 the tiles of a row-major [M, K]
// matrix are consecutive 128-element spans, tile i at x + 128 i with scale
// s[i].  A lane holds one 16-byte vector (EPL elements); LPT lanes cover a
// tile; a warp issues UNROLL vectors per lane before reducing, so each warp
// has UNROLL x 512 B in flight.
template <typename T, int UNROLL>
__global__ void __launch_bounds__(256) act_quant_rows_kernel(const T* __restrict__ x,
                                                             uint8_t* __restrict__ q,
                                                             float* __restrict__ s,
                                                             int64_t n_tiles, int pow2) {
  constexpr int EPL = Vec16<T>::N;            // elements per lane
  constexpr int LPT = 128 / EPL;              // lanes per tile (16 or 32)
  constexpr int TPW = 32 / LPT;               // tiles per warp-vector (2 or 1)
  constexpr int CHUNK = TPW * UNROLL;         // tiles per warp iteration
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int sub = lane % LPT;                 // position inside the tile
  const int tsel = lane / LPT;                // which tile of the warp-vector

  for (int64_t base = warp * CHUNK; base < n_tiles; base += n_warps * CHUNK) {
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t tile = base + u * TPW + tsel;
      v[u] = tile < n_tiles ? ld_stream16(x + tile * 128 + sub * EPL) : make_uint4(0, 0, 0, 0);
    }
    // tile amaxes (every lane of a tile ends with its tile's amax)
    float amax[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float f[EPL];
      Vec16<T>::unpack(v[u], f);
      float a = 0.0f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) a = fmaxf(a, fabsf(f[i]));
#pragma unroll
      for (int off = LPT / 2; off > 0; off >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
      amax[u] = a;
    }
    // lane L < CHUNK derives the scale of tile (u = L / TPW, tile-in-vector
    // L % TPW) once, instead of every lane of every tile doing it
    float my_amax = 0.0f;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const float a = __shfl_sync(0xFFFFFFFFu, amax[u], (lane % TPW) * LPT);
      if (lane / TPW == u) my_amax = a;
    }
    const Scale mine = scale_from_amax(my_amax, pow2 != 0);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t tile = base + u * TPW + tsel;
      float f[EPL];
      Vec16<T>::unpack(v[u], f);
      const int src = u * TPW + tsel;
      const Scale sc = {__shfl_sync(0xFFFFFFFFu, mine.s, src), __shfl_sync(0xFFFFFFFFu, mine.m, src)};
      if (tile < n_tiles) {
        uint32_t packed[EPL / 4];
#pragma unroll
        for (int i = 0; i < EPL / 4; ++i) {
          const uint32_t lo = e4m3x2(__fmul_rn(f[4 * i], sc.m), __fmul_rn(f[4 * i + 1], sc.m));
          const uint32_t hi =
              e4m3x2(__fmul_rn(f[4 * i + 2], sc.m), __fmul_rn(f[4 * i + 3], sc.m));
          packed[i] = lo | (hi << 16);
        }
        uint8_t* dst = q + tile * 128 + sub * EPL;
        if constexpr (EPL == 8) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
        } else {
          *reinterpret_cast<uint32_t*>(dst) = packed[0];
        }
        if (sub == 0) s[tile] = sc.s;
      }
    }
  }
}

// --------------------------------------------------------------------------
// 128x1 tiles along M, transposed output.  Persistent CTAs walk blocks of 128
// rows x COLS columns of x (COLS = 128 for BF16, 64 for FP32: 32 KB either
// way); TMA fills a 2-stage ring of such blocks in shared memory, so the
// threads only read columns, convert and store.  The grid is the CTAs of 512
// threads the SMs hold at once (two per SM for BF16, three for FP32).
// Thread (j, g) owns the column
// pair (2j, 2j+1) and rows g*RPG.. of the block: it reads them as 32- or 64-bit
// words (conflict-free: a block row is 256 contiguous bytes), publishes its two
// partial amaxes, and after one barrier reads them again, converts them and
// writes RPG code bytes to each of q^T rows col0+2j and col0+2j+1.
constexpr int kColStages = 2;
constexpr int kColThreads = 512;

template <typename T>
struct ColTile {
  static constexpr int ROWS = 128;
  static constexpr int COLS = sizeof(T) == 2 ? 128 : 64;
  static constexpr int BYTES = ROWS * COLS * static_cast<int>(sizeof(T));
};

template <typename T>
__global__ void __launch_bounds__(kColThreads) act_quant_cols_kernel(const __grid_constant__ CUtensorMap tmX,
                                                             uint8_t* __restrict__ qt,
                                                             float* __restrict__ st, int M, int K,
                                                             int pow2, long long wait_limit,
                                                             int* status) {
  constexpr int ROWS = ColTile<T>::ROWS;
  constexpr int COLS = ColTile<T>::COLS;
  constexpr int NPAIR = COLS / 2;             // column pairs
  constexpr int RG = kColThreads / NPAIR;     // row groups (8 or 16)
  constexpr int RPG = ROWS / RG;              // rows per group (16 or 8)
  extern __shared__ __align__(128) uint8_t qc_smem[];
  T (*tiles)[ROWS][COLS] = reinterpret_cast<T (*)[ROWS][COLS]>(qc_smem);
  __shared__ __align__(8) uint64_t full[kColStages];
  __shared__ float part[RG][COLS];
  __shared__ float colm[COLS];                                          // per-column multipliers
  __shared__ __align__(16) uint8_t codes[RPG == 16 ? COLS : 1][128];   // BF16 path: staged q^T rows
  __shared__ int abort_flag;

  const int t = threadIdx.x;
  const int col_tiles = K / COLS;
  const int n_tiles = col_tiles * (M / ROWS);
  if (t == 0) {
    for (int s = 0; s < kColStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
    abort_flag = 0;
    tma_prefetch_desc(&tmX);
    for (int s = 0; s < kColStages; ++s) {
      const int tile = blockIdx.x + s * gridDim.x;
      if (tile < n_tiles) {
        mbar_arrive_expect_tx(smem_u32(&full[s]), ColTile<T>::BYTES);
        tma_load_2d(smem_u32(&tiles[s][0][0]), &tmX, smem_u32(&full[s]), (tile % col_tiles) * COLS,
                    (tile / col_tiles) * ROWS);
      }
    }
  }
  __syncthreads();

  const int j = t % NPAIR, g = t / NPAIR;
  int i = 0;
  for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++i) {
    const int stg = i % kColStages;
    const bool got =
        mbar_wait(smem_u32(&full[stg]), (i / kColStages) & 1, wait_limit, &abort_flag, status);
    if (__syncthreads_or(!got)) break;
    const int col0 = (tile % col_tiles) * COLS;
    const int rb = tile / col_tiles;
    const int row0 = rb * ROWS;
    T (*blk)[COLS] = tiles[stg];
    // the column pair (2j, 2j+1) at row r of this thread's group
    auto pair_at = [&](int r, float& x0, float& x1) {
      if constexpr (sizeof(T) == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(&blk[g * RPG + r][2 * j]);
        x0 = __uint_as_float(w << 16);
        x1 = __uint_as_float(w & 0xFFFF0000u);
      } else {
        const float2 w = *reinterpret_cast<const float2*>(&blk[g * RPG + r][2 * j]);
        x0 = w.x;
        x1 = w.y;
      }
    };
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int r = 0; r < RPG; ++r) {
      float x0, x1;
      pair_at(r, x0, x1);
      a0 = fmaxf(a0, fabsf(x0));
      a1 = fmaxf(a1, fabsf(x1));
    }
    part[g][2 * j] = a0;
    part[g][2 * j + 1] = a1;
    __syncthreads();
    // one thread per column folds the partials and derives the scale once
    if (t < COLS) {
      float a = part[0][t];
#pragma unroll
      for (int k = 1; k < RG; ++k) a = fmaxf(a, part[k][t]);
      const Scale sc = scale_from_amax(a, pow2 != 0);
      colm[t] = sc.m;
      st[static_cast<int64_t>(col0 + t) * (M / ROWS) + rb] = sc.s;
    }
    __syncthreads();
    const Scale s0 = {0.0f, colm[2 * j]};
    const Scale s1 = {0.0f, colm[2 * j + 1]};
    uint32_t w0[RPG / 4], w1[RPG / 4];
#pragma unroll
    for (int q4 = 0; q4 < RPG / 4; ++q4) {
      float x[4], y[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pair_at(4 * q4 + e, x[e], y[e]);
      w0[q4] = e4m3x2(__fmul_rn(x[0], s0.m), __fmul_rn(x[1], s0.m)) |
               (e4m3x2(__fmul_rn(x[2], s0.m), __fmul_rn(x[3], s0.m)) << 16);
      w1[q4] = e4m3x2(__fmul_rn(y[0], s1.m), __fmul_rn(y[1], s1.m)) |
               (e4m3x2(__fmul_rn(y[2], s1.m), __fmul_rn(y[3], s1.m)) << 16);
    }
    if constexpr (RPG == 16) {
      // Stage the codes as q^T rows (128 bytes each) in shared memory, 16-byte
      // chunk c of row k at position c ^ ((k / 2) % 8): the chunk writes below
      // and the row reads of the copy-out both use every bank once per
      // 128-byte wavefront.  The copy-out then writes whole 128-byte lines.
      *reinterpret_cast<uint4*>(&codes[2 * j][16 * (g ^ (j % 8))]) =
          make_uint4(w0[0], w0[1], w0[2], w0[3]);
      *reinterpret_cast<uint4*>(&codes[2 * j + 1][16 * (g ^ (j % 8))]) =
          make_uint4(w1[0], w1[1], w1[2], w1[3]);
      __syncthreads();
#pragma unroll
      for (int q16 = 0; q16 < COLS * 8 / kColThreads; ++q16) {
        const int ci = t + kColThreads * q16;
        const int k = ci / 8, c = ci % 8;
        const uint4 v = *reinterpret_cast<const uint4*>(&codes[k][16 * (c ^ ((k / 2) % 8))]);
        *reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + k) * M + row0 + 16 * c) = v;
      }
    } else {
      uint8_t* d0 = qt + static_cast<int64_t>(col0 + 2 * j) * M + row0 + g * RPG;
      uint8_t* d1 = qt + static_cast<int64_t>(col0 + 2 * j + 1) * M + row0 + g * RPG;
      *reinterpret_cast<uint2*>(d0) = make_uint2(w0[0], w0[1]);
      *reinterpret_cast<uint2*>(d1) = make_uint2(w1[0], w1[1]);
    }
    // every thread is done with this stage, part[] and codes[]: refill it
    __syncthreads();
    if (t == 0) {
      const int next = tile + kColStages * gridDim.x;
      if (next < n_tiles) {
        mbar_arrive_expect_tx(smem_u32(&full[stg]), ColTile<T>::BYTES);
        tma_load_2d(smem_u32(&tiles[stg][0][0]), &tmX, smem_u32(&full[stg]),
                    (next % col_tiles) * COLS, (next / col_tiles) * ROWS);
      }
    }
  }
  // after an abort, let copies still in flight land before the CTA exits
  if (abort_flag && t == 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < (1 << 20)) __nanosleep(1000);
  }
}

// --------------------------------------------------------------------------
// Backward re-quantisation (page 5, backward-pass passage): stored E4M3 codes
// with 1x128 scales -> dequantise (one FP32 multiply) -> 128x1 tiles with
// transposed output.  One CTA owns rows [128 i, 128 i+128) and the 128 columns
// of one scale group, so each row has a single scale: the 16 KB code block and
// the 128 row scales are staged in shared memory.  Thread (j, g) owns the
// column pair (2j, 2j+1) and rows 32g..32g+31; as in act_quant_cols it takes
// the column amax in a first pass and converts in a second; the codes are then
// staged as q^T rows in shared memory and written as whole 128-byte rows.
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two_codes, float& lo, float& hi) {
  uint32_t h2;   // E4M3 -> FP16 is exact (E4M3 is a subset of FP16)
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two_codes)));
  lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
  hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

__global__ void __launch_bounds__(256) requant_t_kernel(const uint8_t* __restrict__ q,
                                                        const float* __restrict__ s,
                                                        uint8_t* __restrict__ qt,
                                                        float* __restrict__ st, int M, int K,
                                                        int pow2) {
  constexpr int ROWS = 128, COLS = 128, RPG = 32;
  __shared__ __align__(16) uint8_t tile[ROWS][COLS];
  __shared__ float rs[ROWS];
  __shared__ float part[4][COLS];
  const int row0 = blockIdx.y * ROWS;
  const int col0 = blockIdx.x * COLS;
  const int nkg = K / 128;
  const int t = threadIdx.x;

  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vid = t + 256 * i;
    const int r = vid / 8, c = (vid % 8) * 16;
    v[i] = ld_stream16(q + static_cast<int64_t>(row0 + r) * K + col0 + c);
  }
  if (t < ROWS) rs[t] = __ldg(s + static_cast<int64_t>(row0 + t) * nkg + blockIdx.x);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int vid = t + 256 * i;
    *reinterpret_cast<uint4*>(&tile[vid / 8][(vid % 8) * 16]) = v[i];
  }
  __syncthreads();

  const int j = t % 64, g = t / 64;
  auto pair_at = [&](int r, float& x0, float& x1) {
    const int row = g * RPG + r;
    const uint32_t two = *reinterpret_cast<const uint16_t*>(&tile[row][2 * j]);
    float d0, d1;
    e4m3x2_to_f32(two, d0, d1);
    const float sc = rs[row];
    x0 = __fmul_rn(d0, sc);
    x1 = __fmul_rn(d1, sc);
  };
  float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 8
  for (int r = 0; r < RPG; ++r) {
    float x0, x1;
    pair_at(r, x0, x1);
    a0 = fmaxf(a0, fabsf(x0));
    a1 = fmaxf(a1, fabsf(x1));
  }
  part[g][2 * j] = a0;
  part[g][2 * j + 1] = a1;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a0 = fmaxf(a0, part[i][2 * j]);
    a1 = fmaxf(a1, part[i][2 * j + 1]);
  }
  const Scale s0 = scale_from_amax(a0, pow2 != 0);
  const Scale s1 = scale_from_amax(a1, pow2 != 0);
  if (g == 0) {
    st[static_cast<int64_t>(col0 + 2 * j) * (M / ROWS) + blockIdx.y] = s0.s;
    st[static_cast<int64_t>(col0 + 2 * j + 1) * (M / ROWS) + blockIdx.y] = s1.s;
  }
  uint32_t w0[RPG / 4], w1[RPG / 4];
#pragma unroll
  for (int i = 0; i < RPG / 4; ++i) {
    float x[4], y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pair_at(4 * i + e, x[e], y[e]);
    w0[i] = e4m3x2(__fmul_rn(x[0], s0.m), __fmul_rn(x[1], s0.m)) |
            (e4m3x2(__fmul_rn(x[2], s0.m), __fmul_rn(x[3], s0.m)) << 16);
    w1[i] = e4m3x2(__fmul_rn(y[0], s1.m), __fmul_rn(y[1], s1.m)) |
            (e4m3x2(__fmul_rn(y[2], s1.m), __fmul_rn(y[3], s1.m)) << 16);
  }
  // stage the codes as q^T rows in the (no longer needed) code tile, 16-byte
  // chunk c of row k at position c ^ ((k / 2) % 8), then write whole rows
  __syncthreads();
  uint8_t (*out)[COLS] = tile;
  const int sw = j % 8;
  *reinterpret_cast<uint4*>(&out[2 * j][16 * ((2 * g) ^ sw)]) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
  *reinterpret_cast<uint4*>(&out[2 * j][16 * ((2 * g + 1) ^ sw)]) =
      make_uint4(w0[4], w0[5], w0[6], w0[7]);
  *reinterpret_cast<uint4*>(&out[2 * j + 1][16 * ((2 * g) ^ sw)]) =
      make_uint4(w1[0], w1[1], w1[2], w1[3]);
  *reinterpret_cast<uint4*>(&out[2 * j + 1][16 * ((2 * g + 1) ^ sw)]) =
      make_uint4(w1[4], w1[5], w1[6], w1[7]);
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ci = t + 256 * i;
    const int k = ci / 8, c = ci % 8;
    const uint4 v = *reinterpret_cast<const uint4*>(&out[k][16 * (c ^ ((k / 2) % 8))]);
    *reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + k) * M + row0 + 16 * c) = v;
  }
}

// --------------------------------------------------------------------------
// 128x128 blocks.  One CTA per block: load the block into registers while
// reducing the amax, then write row-major codes (8 bytes per lane, coalesced)
// and, if requested, the transposed codes: then the block is also staged in
// shared memory, and thread (j, g) reads columns 2j, 2j+1 of rows
// 32g..32g+31 and writes 32 bytes of each of q^T rows 2j and 2j+1.  The
// kernel is bound by how many loads are in flight, so a BF16 block is held
// in at most 64 registers per thread: four CTAs per SM instead of two
// (18432 x 7168: 77.8 -> 65.5 us).  FP32 blocks keep two CTAs per SM (at 64
// registers they would spill).
template <typename T>
__global__ void __launch_bounds__(256, sizeof(T) == 2 ? 4 : 2) weight_quant_kernel(const T* __restrict__ w,
                                                           uint8_t* __restrict__ q,
                                                           float* __restrict__ s,
                                                           uint8_t* __restrict__ qt,
                                                           float* __restrict__ st, int N, int K,
                                                           int pow2) {
  constexpr int B = 128;
  constexpr int EPV = Vec16<T>::N;
  constexpr int VPR = B / EPV;                 // vectors per block row
  constexpr int NV = B * VPR / 256;            // vectors per thread
  extern __shared__ __align__(16) uint8_t wq_smem[];
  T (*blk)[B] = reinterpret_cast<T (*)[B]>(wq_smem);   // [128][128] of T (32 or 64 KB)
  __shared__ float red[8];

  const int bn = blockIdx.y, bk = blockIdx.x;
  const int row0 = bn * B, col0 = bk * B;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;

  uint4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vid = t + 256 * i;
    const int r = vid / VPR, c = (vid % VPR) * EPV;
    v[i] = ld_stream16(w + static_cast<int64_t>(row0 + r) * K + col0 + c);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vid = t + 256 * i;
    const int r = vid / VPR, c = (vid % VPR) * EPV;
    if (qt != nullptr) *reinterpret_cast<uint4*>(&blk[r][c]) = v[i];
    float f[EPV];
    Vec16<T>::unpack(v[i], f);
#pragma unroll
    for (int e = 0; e < EPV; ++e) amax = fmaxf(amax, fabsf(f[e]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const Scale sc = scale_from_amax(amax, pow2 != 0);
  if (t == 0) {
    s[bn * (K / B) + bk] = sc.s;
    if (st != nullptr) st[bk * (N / B) + bn] = sc.s;
  }

  // row-major codes, straight from the registers
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vid = t + 256 * i;
    const int r = vid / VPR, c = (vid % VPR) * EPV;
    float f[EPV];
    Vec16<T>::unpack(v[i], f);
    uint32_t packed[EPV / 4];
#pragma unroll
    for (int e = 0; e < EPV / 4; ++e) {
      const uint32_t lo = e4m3x2(__fmul_rn(f[4 * e], sc.m), __fmul_rn(f[4 * e + 1], sc.m));
      const uint32_t hi = e4m3x2(__fmul_rn(f[4 * e + 2], sc.m), __fmul_rn(f[4 * e + 3], sc.m));
      packed[e] = lo | (hi << 16);
    }
    uint8_t* dst = q + static_cast<int64_t>(row0 + r) * K + col0 + c;
    if constexpr (EPV == 8) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = packed[0];
    }
  }

  if (qt != nullptr) {
    // thread (j, g): columns 2j, 2j+1 of the block, rows 32g..32g+31, read as
    // one 32- or 64-bit shared word per row (conflict-free)
    const int j = t % 64, g = t / 64;
    uint32_t w0[8], w1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float x[4], y[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = 32 * g + 4 * i + e;
        if constexpr (sizeof(T) == 2) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(&blk[r][2 * j]);
          x[e] = __uint_as_float(w << 16);
          y[e] = __uint_as_float(w & 0xFFFF0000u);
        } else {
          const float2 w = *reinterpret_cast<const float2*>(&blk[r][2 * j]);
          x[e] = w.x;
          y[e] = w.y;
        }
      }
      w0[i] = e4m3x2(__fmul_rn(x[0], sc.m), __fmul_rn(x[1], sc.m)) |
              (e4m3x2(__fmul_rn(x[2], sc.m), __fmul_rn(x[3], sc.m)) << 16);
      w1[i] = e4m3x2(__fmul_rn(y[0], sc.m), __fmul_rn(y[1], sc.m)) |
              (e4m3x2(__fmul_rn(y[2], sc.m), __fmul_rn(y[3], sc.m)) << 16);
    }
    // stage the codes as q^T rows in the block's shared memory (no longer
    // read), 16-byte chunk c of row k at position c ^ ((k / 2) % 8), then
    // write whole 128-byte rows of q^T
    __syncthreads();
    uint8_t (*out)[B] = reinterpret_cast<uint8_t (*)[B]>(wq_smem);
    const int sw = j % 8;
    *reinterpret_cast<uint4*>(&out[2 * j][16 * ((2 * g) ^ sw)]) =
        make_uint4(w0[0], w0[1], w0[2], w0[3]);
    *reinterpret_cast<uint4*>(&out[2 * j][16 * ((2 * g + 1) ^ sw)]) =
        make_uint4(w0[4], w0[5], w0[6], w0[7]);
    *reinterpret_cast<uint4*>(&out[2 * j + 1][16 * ((2 * g) ^ sw)]) =
        make_uint4(w1[0], w1[1], w1[2], w1[3]);
    *reinterpret_cast<uint4*>(&out[2 * j + 1][16 * ((2 * g + 1) ^ sw)]) =
        make_uint4(w1[4], w1[5], w1[6], w1[7]);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ci = t + 256 * i;
      const int k = ci / 8, c = ci % 8;
      const uint4 v = *reinterpret_cast<const uint4*>(&out[k][16 * (c ^ ((k / 2) % 8))]);
      *reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + k) * N + row0 + 16 * c) = v;
    }
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers
cudaError_t launch_act_quant_rows(const void* x, fp8fg_dtype xt, int64_t M, int64_t K, uint8_t* q,
                                  float* s, bool pow2, cudaStream_t st) {
  const int64_t n_tiles = M * (K / 128);
  const int sms = device_sm_count();
  constexpr int kUnroll = 4;
  const int tiles_per_block = (xt == FP8FG_BF16 ? 2 : 1) * kUnroll * 8;  // 8 warps
  int64_t blocks = (n_tiles + tiles_per_block - 1) / tiles_per_block;
  blocks = blocks < static_cast<int64_t>(sms) * 8 ? blocks : static_cast<int64_t>(sms) * 8;
  if (blocks < 1) blocks = 1;
  if (xt == FP8FG_BF16)
    act_quant_rows_kernel<__nv_bfloat16, kUnroll><<<static_cast<int>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), q, s, n_tiles, pow2 ? 1 : 0);
  else
    act_quant_rows_kernel<float, kUnroll><<<static_cast<int>(blocks), 256, 0, st>>>(
        static_cast<const float*>(x), q, s, n_tiles, pow2 ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_act_quant_cols(const void* x, fp8fg_dtype xt, int64_t M, int64_t K, uint8_t* qt,
                                  float* st_, bool pow2, cudaStream_t st) {
  const bool bf16 = xt == FP8FG_BF16;
  const int cols = bf16 ? ColTile<__nv_bfloat16>::COLS : ColTile<float>::COLS;
  const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
  const uint64_t strides[1] = {static_cast<uint64_t>(K) * (bf16 ? 2 : 4)};
  const uint32_t box[2] = {static_cast<uint32_t>(cols), 128};
  CUtensorMap map;
  if (!encode_tensor_map(&map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         x, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const int64_t n_tiles = (K / cols) * (M / 128);
  const int smem = kColStages * 32768;
  // persistent: exactly the CTAs the SMs hold at once (two per SM with the
  // 64 KB ring and the static staging), so that no CTA waits for an SM
  const cudaError_t attr = bf16 ? set_max_dynamic_smem<act_quant_cols_kernel<__nv_bfloat16>>(smem)
                                : set_max_dynamic_smem<act_quant_cols_kernel<float>>(smem);
  if (attr != cudaSuccess) return attr;
  const int per_sm = bf16 ? resident_ctas_per_sm<act_quant_cols_kernel<__nv_bfloat16>>(kColThreads, smem)
                          : resident_ctas_per_sm<act_quant_cols_kernel<float>>(kColThreads, smem);
  const int64_t max_ctas = static_cast<int64_t>(device_sm_count()) * per_sm;
  const int grid = static_cast<int>(n_tiles < max_ctas ? n_tiles : max_ctas);
  if (bf16)
    act_quant_cols_kernel<__nv_bfloat16><<<grid, kColThreads, smem, st>>>(
        map, qt, st_, static_cast<int>(M), static_cast<int>(K), pow2 ? 1 : 0, wait_limit_cycles(),
        device_status_word());
  else
    act_quant_cols_kernel<float><<<grid, kColThreads, smem, st>>>(
        map, qt, st_, static_cast<int>(M), static_cast<int>(K), pow2 ? 1 : 0, wait_limit_cycles(),
        device_status_word());
  return cudaGetLastError();
}

cudaError_t launch_requant_t(const uint8_t* q, const float* s, int64_t M, int64_t K, uint8_t* qt,
                             float* st_, bool pow2, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(M / 128));
  requant_t_kernel<<<grid, 256, 0, st>>>(q, s, qt, st_, static_cast<int>(M), static_cast<int>(K),
                                         pow2 ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_weight_quant(const void* w, fp8fg_dtype wt, int64_t N, int64_t K, uint8_t* q,
                                float* s, uint8_t* qt, float* st_, bool pow2, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(N / 128));
  // shared memory only for the transposed copy
  if (wt == FP8FG_BF16) {
    const int smem = qt != nullptr ? 128 * 128 * 2 : 0;
    weight_quant_kernel<__nv_bfloat16><<<grid, 256, smem, st>>>(
        static_cast<const __nv_bfloat16*>(w), q, s, qt, st_, static_cast<int>(N),
        static_cast<int>(K), pow2 ? 1 : 0);
  } else {
    constexpr int smem_max = 128 * 128 * 4;
    const cudaError_t attr = set_max_dynamic_smem<weight_quant_kernel<float>>(smem_max);
    const int smem = qt != nullptr ? smem_max : 0;
    if (attr != cudaSuccess) return attr;
    weight_quant_kernel<float><<<grid, 256, smem, st>>>(static_cast<const float*>(w), q, s, qt,
                                                        st_, static_cast<int>(N),
                                                        static_cast<int>(K), pow2 ? 1 : 0);
  }
  return cudaGetLastError();
}

}  // namespace fp8fg
