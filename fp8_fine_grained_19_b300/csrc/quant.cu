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
// and columns [64 j, 64 j + 64) of x.  The block is staged as float in shared
// memory; each column's amax comes from 4 quarter-column partials; then thread
// (k, p) converts rows 32p..32p+31 of column k and writes 32 consecutive code
// bytes of q^T row k (a full 32-byte sector).
template <typename T>
__global__ void __launch_bounds__(256) act_quant_cols_kernel(const T* __restrict__ x,
                                                             uint8_t* __restrict__ qt,
                                                             float* __restrict__ st, int M,
                                                             int K, int pow2) {
  constexpr int ROWS = 128, COLS = 64;
  constexpr int EPV = Vec16<T>::N;            // elements per 16-byte vector
  constexpr int VPR = COLS / EPV;             // vectors per tile row
  __shared__ __align__(16) float tile[ROWS][COLS];
  __shared__ float part[4][COLS];
  __shared__ float mul[COLS];

  const int row0 = blockIdx.y * ROWS;
  const int col0 = blockIdx.x * COLS;
  const int t = threadIdx.x;

  constexpr int NV = ROWS * VPR / 256;        // vectors per thread
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
    float f[EPV];
    Vec16<T>::unpack(v[i], f);
#pragma unroll
    for (int e = 0; e < EPV; e += 4)
      *reinterpret_cast<float4*>(&tile[r][c + e]) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
  }
  __syncthreads();

  const int k = t % COLS, p = t / COLS;       // column, quarter (32 rows)
  float amax = 0.0f;
#pragma unroll 8
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(tile[32 * p + j][k]));
  part[p][k] = amax;
  __syncthreads();
  if (t < COLS) {
    const float a = fmaxf(fmaxf(part[0][t], part[1][t]), fmaxf(part[2][t], part[3][t]));
    const Scale sc = scale_from_amax(a, pow2 != 0);
    mul[t] = sc.m;
    st[static_cast<int64_t>(col0 + t) * (M / ROWS) + blockIdx.y] = sc.s;
  }
  __syncthreads();

  const float m = mul[k];
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float* r4 = &tile[32 * p + 4 * j][k];
    const uint32_t lo = e4m3x2(__fmul_rn(r4[0], m), __fmul_rn(r4[COLS], m));
    const uint32_t hi = e4m3x2(__fmul_rn(r4[2 * COLS], m), __fmul_rn(r4[3 * COLS], m));
    w[j] = lo | (hi << 16);
  }
  uint4* dst = reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + k) * M + row0 + 32 * p);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// --------------------------------------------------------------------------
// 128x128 blocks.  One CTA per block: stage the block (input type) in shared
// memory while reducing the amax, then write row-major codes (8 bytes per
// lane, coalesced) and, if requested, the transposed codes (thread (k, p)
// walks rows 64p..64p+63 of column k and writes 64 bytes of q^T row k).
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
    const int k = t % B, p = t / B;           // column of the block, half (64 rows)
    uint32_t wv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int r = 64 * p + 4 * j;
      const uint32_t lo = e4m3x2(__fmul_rn(to_f32(blk[r][k]), sc.m),
                                 __fmul_rn(to_f32(blk[r + 1][k]), sc.m));
      const uint32_t hi = e4m3x2(__fmul_rn(to_f32(blk[r + 2][k]), sc.m),
                                 __fmul_rn(to_f32(blk[r + 3][k]), sc.m));
      wv[j] = lo | (hi << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(qt + static_cast<int64_t>(col0 + k) * N + row0 + 64 * p);
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[j] = make_uint4(wv[4 * j], wv[4 * j + 1], wv[4 * j + 2], wv[4 * j + 3]);
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
  const dim3 grid(static_cast<unsigned>(K / 64), static_cast<unsigned>(M / 128));
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
