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

constexpr float kE4M3Max = 448.0f;
constexpr float kAmaxFloor = 5.42101086242752217e-20f;  // 2^-64

struct Scale {
  float s;  // dequantisation scale (stored)
  float m;  // quantisation multiplier
};

__device__ __forceinline__ Scale scale_from_amax(float amax, bool pow2) {
  const float a = fmaxf(amax, kAmaxFloor);
  const float t = __fdiv_rn(a, kE4M3Max);
  if (!pow2) return {t, __fdiv_rn(kE4M3Max, a)};
  // t is a normal float in [2^-73, 2^120]: round up to the next power of two
  const uint32_t bits = __float_as_uint(t);
  int e = static_cast<int>((bits >> 23) & 0xFF) - 127;
  if (bits & 0x7FFFFFu) e += 1;
  return {__uint_as_float(static_cast<uint32_t>(e + 127) << 23),
          __uint_as_float(static_cast<uint32_t>(127 - e) << 23)};
}

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

__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

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
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int64_t tile = base + u * TPW + tsel;
      float f[EPL];
      Vec16<T>::unpack(v[u], f);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
      for (int off = LPT / 2; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      if (tile < n_tiles) {
        const Scale sc = scale_from_amax(amax, pow2 != 0);
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
// 128x1 tiles along M, transposed output.  One CTA owns rows [128 i, 128 i+128)
// and COLS columns of x (COLS = 128 for BF16, 64 for FP32: 32 KB either way),
// staged raw in shared memory by coalesced 16-byte loads.  Thread (j, g) owns
// the column pair (2j, 2j+1) and rows g*RPG.. of the block: it reads them as
// 32- or 64-bit words (conflict-free), publishes its two partial amaxes, and
// after one barrier reads them again, converts them and writes RPG code bytes
// to each of q^T rows col0+2j and col0+2j+1.
template <typename T>
__global__ void __launch_bounds__(256) act_quant_cols_kernel(const T* __restrict__ x,
                                                             uint8_t* __restrict__ qt,
                                                             float* __restrict__ st, int M,
                                                             int K, int pow2) {
  constexpr int ROWS = 128;
  constexpr int COLS = sizeof(T) == 2 ? 128 : 64;
  constexpr int EPV = Vec16<T>::N;            // elements per 16-byte vector
  constexpr int VPR = COLS / EPV;             // vectors per tile row (16)
  constexpr int NV = ROWS * VPR / 256;        // vectors per thread (8)
  constexpr int NPAIR = COLS / 2;             // column pairs
  constexpr int RG = 256 / NPAIR;             // row groups (4 or 8)
  constexpr int RPG = ROWS / RG;              // rows per group (32 or 16)
  __shared__ __align__(16) T tile[ROWS][COLS];
  __shared__ float part[RG][COLS];

  const int row0 = blockIdx.y * ROWS;
  const int col0 = blockIdx.x * COLS;
  const int t = threadIdx.x;

  uint4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vid = t + 256 * i;
    const int r = vid / VPR, c = (vid % VPR) * EPV;
    v[i] = ld_stream16(x + static_cast<int64_t>(row0 + r) * K + col0 + c);
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vid = t + 256 * i;
    const int r = vid / VPR, c = (vid % VPR) * EPV;
    *reinterpret_cast<uint4*>(&tile[r][c]) = v[i];
  }
  __syncthreads();

  const int j = t % NPAIR, g = t / NPAIR;
  // the column pair (2j, 2j+1) at row r of this thread's group
  auto pair_at = [&](int r, float& x0, float& x1) {
    if constexpr (sizeof(T) == 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(&tile[g * RPG + r][2 * j]);
      x0 = __uint_as_float(w << 16);
      x1 = __uint_as_float(w & 0xFFFF0000u);
    } else {
      const float2 w = *reinterpret_cast<const float2*>(&tile[g * RPG + r][2 * j]);
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
#pragma unroll
  for (int i = 0; i < RG; ++i) {
    a0 = fmaxf(a0, part[i][2 * j]);
    a1 = fmaxf(a1, part[i][2 * j + 1]);
  }
  const Scale s0 = scale_from_amax(a0, pow2 != 0);
  const Scale s1 = scale_from_amax(a1, pow2 != 0);
  if (g == 0) {
    st[static_cast<int64_t>(col0 + 2 * j) * (M / ROWS) + blockIdx.y] = s0.s;
    st[static_cast<int64_t>(col0 + 2 * j + 1) * (M / ROWS) + blockIdx.y] = s1.s;
  }
  // second pass over the same shared words (cheaper than holding 2 x RPG
  // values in registers, which would cap the CTAs per SM)
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
  uint4* d0 = reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + 2 * j) * M + row0 + g * RPG);
  uint4* d1 = reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + 2 * j + 1) * M + row0 + g * RPG);
#pragma unroll
  for (int i = 0; i < RPG / 16; ++i) {
    d0[i] = make_uint4(w0[4 * i], w0[4 * i + 1], w0[4 * i + 2], w0[4 * i + 3]);
    d1[i] = make_uint4(w1[4 * i], w1[4 * i + 1], w1[4 * i + 2], w1[4 * i + 3]);
  }
}

// --------------------------------------------------------------------------
// Backward re-quantisation (page 5, backward-pass passage): stored E4M3 codes
// with 1x128 scales -> dequantise (one FP32 multiply) -> 128x1 tiles with
// transposed output.  One CTA owns rows [128 i, 128 i+128) and the 128 columns
// of one scale group, so each row has a single scale: the 16 KB code block and
// the 128 row scales are staged in shared memory.  Thread (j, g) owns the
// column pair (2j, 2j+1) and rows 32g..32g+31; as in act_quant_cols it takes
// the column amax in a first pass and converts in a second, writing 32 code
// bytes to each of q^T rows col0+2j and col0+2j+1.
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
  uint4* d0 = reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + 2 * j) * M + row0 + g * RPG);
  uint4* d1 = reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + 2 * j + 1) * M + row0 + g * RPG);
  d0[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
  d0[1] = make_uint4(w0[4], w0[5], w0[6], w0[7]);
  d1[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  d1[1] = make_uint4(w1[4], w1[5], w1[6], w1[7]);
}

// --------------------------------------------------------------------------
// 128x128 blocks.  One CTA per block: stage the block (input type) in shared
// memory while reducing the amax, then write row-major codes (8 bytes per
// lane, coalesced) and, if requested, the transposed codes (thread (j, g)
// reads columns 2j, 2j+1 of rows 32g..32g+31 and writes 32 bytes of each of
// q^T rows 2j and 2j+1).
template <typename T>
__global__ void __launch_bounds__(256) weight_quant_kernel(const T* __restrict__ w,
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
    *reinterpret_cast<uint4*>(&blk[r][c]) = v[i];
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
    uint4* d0 = reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + 2 * j) * N + row0 + 32 * g);
    uint4* d1 =
        reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + 2 * j + 1) * N + row0 + 32 * g);
    d0[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
    d0[1] = make_uint4(w0[4], w0[5], w0[6], w0[7]);
    d1[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
    d1[1] = make_uint4(w1[4], w1[5], w1[6], w1[7]);
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
  const unsigned cols = xt == FP8FG_BF16 ? 128 : 64;    // columns per CTA (K % 128 == 0)
  const dim3 grid(static_cast<unsigned>(K / cols), static_cast<unsigned>(M / 128));
  if (xt == FP8FG_BF16)
    act_quant_cols_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), qt, st_, static_cast<int>(M), static_cast<int>(K),
        pow2 ? 1 : 0);
  else
    act_quant_cols_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), qt, st_,
                                                       static_cast<int>(M), static_cast<int>(K),
                                                       pow2 ? 1 : 0);
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
  if (wt == FP8FG_BF16) {
    constexpr int smem = 128 * 128 * 2;
    weight_quant_kernel<__nv_bfloat16><<<grid, 256, smem, st>>>(
        static_cast<const __nv_bfloat16*>(w), q, s, qt, st_, static_cast<int>(N),
        static_cast<int>(K), pow2 ? 1 : 0);
  } else {
    constexpr int smem = 128 * 128 * 4;
    static const cudaError_t attr = cudaFuncSetAttribute(
        weight_quant_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (attr != cudaSuccess) return attr;
    weight_quant_kernel<float><<<grid, 256, smem, st>>>(static_cast<const float*>(w), q, s, qt,
                                                        st_, static_cast<int>(N),
                                                        static_cast<int>(K), pow2 ? 1 : 0);
  }
  return cudaGetLastError();
}

}  // namespace fp8fg
