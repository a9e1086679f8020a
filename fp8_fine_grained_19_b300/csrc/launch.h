// Internal launcher declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8fg.h"

#include <atomic>

namespace fp8fg {

// Devices the per-device caches below can track (device indices 0 .. 63).
constexpr int kMaxDevices = 64;

// Index of the calling thread's current device, or -1 (no device, or >= kMaxDevices).
int current_device();
// Number of SMs of the current device (cached per device).
int device_sm_count();
// Cycle limit applied to every pipeline wait of the next launches.
long long wait_limit_cycles();
// Device address of the library status word on the current device.
int* device_status_word();

cudaError_t launch_act_quant_rows(const void* x, fp8fg_dtype xt, int64_t M, int64_t K, uint8_t* q,
                                  float* s, bool pow2, cudaStream_t st);
cudaError_t launch_act_quant_cols(const void* x, fp8fg_dtype xt, int64_t M, int64_t K, uint8_t* qt,
                                  float* st_, bool pow2, cudaStream_t st);
cudaError_t launch_requant_t(const uint8_t* q, const float* s, int64_t M, int64_t K, uint8_t* qt,
                             float* st_, bool pow2, cudaStream_t st);
cudaError_t launch_weight_quant(const void* w, fp8fg_dtype wt, int64_t N, int64_t K, uint8_t* q,
                                float* s, uint8_t* qt, float* st_, bool pow2, cudaStream_t st);

// Dense block-scaled GEMM (b_tile: B carries 1x128 tile scales).
// whole_k: study mode, all of K accumulated in the tensor core, per-tensor scales.
// ws / ws_bytes: optional stream-K workspace (used when at least
// gemm_workspace_bytes(...) bytes); force_sk splits even when it would not pay.
fp8fg_status launch_gemm(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                         void* c, fp8fg_dtype ct, int64_t M, int64_t N, int64_t K, bool b_tile,
                         bool whole_k, void* ws, size_t ws_bytes, bool force_sk, cudaStream_t st);
// Workspace a stream-K split of this dense GEMM needs on the current device (0: not split).
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, bool whole_k, bool force_sk);
// launch_gemm with the split's partial tiles in the library's own device array
// (no caller workspace); FP8FG_ERR_UNSUPPORTED_SHAPE when the split needs more.
fp8fg_status launch_gemm_noalloc(const uint8_t* a, const float* sa, const uint8_t* b,
                                 const float* sb, void* c, fp8fg_dtype ct, int64_t M, int64_t N,
                                 int64_t K, bool b_tile, bool force_sk, cudaStream_t st);
// Dense block-scaled GEMM whose result leaves as 1x128 E4M3 tiles (q, s).
fp8fg_status launch_gemm_quant(const uint8_t* a, const float* sa, const uint8_t* b,
                               const float* sb, uint8_t* q, float* s, int64_t M, int64_t N,
                               int64_t K, bool b_tile, bool pow2, cudaStream_t st);
// Grouped block-scaled GEMM over contiguous expert row groups.
fp8fg_status launch_grouped_gemm(const uint8_t* a, const float* sa, const int32_t* offsets,
                                 int32_t E, int64_t total_rows, const uint8_t* b, const float* sb,
                                 void* c, fp8fg_dtype ct, int64_t N, int64_t K, cudaStream_t st);
// Grouped up-projection with SwiGLU; h leaves as 1x128 E4M3 tiles (q, s).
fp8fg_status launch_grouped_swiglu_quant(const uint8_t* a, const float* sa,
                                         const int32_t* offsets, int32_t E, int64_t total_rows,
                                         const uint8_t* b, const float* sb, uint8_t* q, float* s,
                                         int64_t N, int64_t K, bool pow2, cudaStream_t st);
// Failure-detection self-test: one wait that nothing completes.
cudaError_t launch_wait_timeout_selftest(uint32_t limit_cycles, cudaStream_t st);

// Raise kernel `Kernel`'s dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the device's context, so it is set once per
// device (and again if a previous attempt failed), not once per process.
template <auto Kernel>
cudaError_t set_max_dynamic_smem(int bytes) {
  static std::atomic<int> done[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0) return cudaErrorInvalidDevice;
  if (done[d].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[d].store(1, std::memory_order_release);
  return e;
}

// CTAs of `Kernel` that one SM of the current device holds at once, launched
// with `threads` threads and `smem` bytes of dynamic shared memory (each kernel
// is always launched with one such shape); at least 1, cached per device.  A
// persistent grid larger than this would leave its last CTAs waiting for SMs.
template <auto Kernel>
int resident_ctas_per_sm(int threads, int smem) {
  static std::atomic<int> cache[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0) return 1;
  int occ = cache[d].load(std::memory_order_acquire);
  if (occ > 0) return occ;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, Kernel, threads, smem) != cudaSuccess ||
      occ < 1)
    occ = 1;
  cache[d].store(occ, std::memory_order_release);
  return occ;
}

// Encode a tensor map (innermost dimension first, zero fill); returns false if
// the driver rejects it.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle);
// The same for uint8 elements with 128-byte swizzling (GEMM operand tiles).
bool encode_tensor_map_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace fp8fg
