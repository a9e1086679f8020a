// C ABI of libfp8fg.so (declared in include/fp8fg.h).
//
// Host side only: argument validation (every rule is checked before any CUDA
// call, so a rejected call never touches the device), launch dispatch, the
// tensor-map encoder (fetched from the driver through the runtime, so the
// library does not link libcuda), the per-device SM-count cache and the
// device status word.

#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "launch.h"

namespace fp8fg {

// Library status word, one per device context (see fp8_get_device_status).
__device__ int g_device_status = 0;

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
constexpr uint64_t kDefaultWaitLimit = uint64_t{1} << 32;  // ~2 s at 2 GHz

std::atomic<uint64_t> g_wait_limit{0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

}  // namespace

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

int device_sm_count() {
  static std::atomic<int> cache[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0) return 0;
  int v = cache[d].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || v <= 0)
    return 0;
  cache[d].store(v, std::memory_order_relaxed);
  return v;
}

int* device_status_word() {
  static std::atomic<int*> cache[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0) return nullptr;
  int* p = cache[d].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return nullptr;
  p = static_cast<int*>(addr);
  cache[d].store(p, std::memory_order_release);
  return p;
}

long long wait_limit_cycles() {
  uint64_t v = g_wait_limit.load(std::memory_order_relaxed);
  if (v == 0) {
    static const uint64_t from_env = [] {
      const char* e = std::getenv("FP8FG_WAIT_LIMIT_CYCLES");
      if (e == nullptr) return uint64_t{0};
      return static_cast<uint64_t>(std::strtoull(e, nullptr, 10));
    }();
    v = from_env ? from_env : kDefaultWaitLimit;
  }
  if (v > (uint64_t{1} << 62)) v = uint64_t{1} << 62;
  return static_cast<long long>(v);
}

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides_bytes[i];
  const CUresult r = enc(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s,
                         b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tensor_map_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rank, dims, strides_bytes,
                           box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace fp8fg

using namespace fp8fg;

namespace {

bool valid_dtype(fp8fg_dtype t) { return t == FP8FG_BF16 || t == FP8FG_F32; }

fp8fg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FP8FG_OK : FP8FG_ERR_CUDA; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Device is usable: fails (FP8FG_ERR_CUDA) without a CUDA device.
bool have_device() { return device_sm_count() > 0; }

}  // namespace

extern "C" {

int fp8fg_abi_version(void) { return 6; }

const char* fp8fg_status_string(fp8fg_status status) {
  switch (status) {
    case FP8FG_OK: return "ok";
    case FP8FG_ERR_INVALID_ARG: return "invalid argument";
    case FP8FG_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case FP8FG_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FP8FG_ERR_CUDA: return "CUDA error (no device, or a failed call or launch)";
    case FP8FG_ERR_TIMEOUT: return "device pipeline wait exceeded its cycle limit";
    case FP8FG_ERR_BAD_OFFSETS: return "expert offsets are not 0..total_rows non-decreasing";
  }
  return "unknown status";
}

void fp8fg_set_wait_limit(uint64_t cycles) { g_wait_limit.store(cycles); }

fp8fg_status fp8_act_quant(const void* x, fp8fg_dtype x_dtype, int64_t M, int64_t K, uint8_t* q,
                           float* s, unsigned flags, void* stream) {
  if (!valid_dtype(x_dtype) || (flags & ~(FP8FG_POW2 | FP8FG_TRANSPOSE)) != 0 || M < 0 || K < 0)
    return FP8FG_ERR_INVALID_ARG;
  if (M > 0 && (x == nullptr || q == nullptr || s == nullptr)) return FP8FG_ERR_INVALID_ARG;
  if (K < 128 || K % 128 != 0 || M > kMaxDim || K > kMaxDim) return FP8FG_ERR_UNSUPPORTED_SHAPE;
  const bool trans = (flags & FP8FG_TRANSPOSE) != 0;
  if (trans && (M % 128 != 0 || M / 128 > 65535)) return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s)) return FP8FG_ERR_MISALIGNED;
  if (M == 0) return FP8FG_OK;
  if (!have_device()) return FP8FG_ERR_CUDA;
  const bool pow2 = (flags & FP8FG_POW2) != 0;
  if (trans) return from_cuda(launch_act_quant_cols(x, x_dtype, M, K, q, s, pow2, as_stream(stream)));
  return from_cuda(launch_act_quant_rows(x, x_dtype, M, K, q, s, pow2, as_stream(stream)));
}

fp8fg_status fp8_requant_transpose(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                   uint8_t* q_t, float* s_t, unsigned flags, void* stream) {
  if ((flags & ~FP8FG_POW2) != 0 || M < 0 || K < 0) return FP8FG_ERR_INVALID_ARG;
  if (M > 0 && (q == nullptr || s == nullptr || q_t == nullptr || s_t == nullptr))
    return FP8FG_ERR_INVALID_ARG;
  if (K < 128 || K % 128 != 0 || M % 128 != 0 || M > kMaxDim || K > kMaxDim ||
      M / 128 > 65535)
    return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(q) || !aligned16(s) || !aligned16(q_t) || !aligned16(s_t))
    return FP8FG_ERR_MISALIGNED;
  if (M == 0) return FP8FG_OK;
  if (!have_device()) return FP8FG_ERR_CUDA;
  return from_cuda(launch_requant_t(q, s, M, K, q_t, s_t, (flags & FP8FG_POW2) != 0,
                                    as_stream(stream)));
}

fp8fg_status fp8_weight_quant(const void* w, fp8fg_dtype w_dtype, int64_t N, int64_t K, uint8_t* q,
                              float* s, uint8_t* q_t, float* s_t, unsigned flags, void* stream) {
  if (!valid_dtype(w_dtype) || (flags & ~FP8FG_POW2) != 0 || N < 0 || K < 0)
    return FP8FG_ERR_INVALID_ARG;
  if (w == nullptr || q == nullptr || s == nullptr || ((q_t == nullptr) != (s_t == nullptr)))
    return FP8FG_ERR_INVALID_ARG;
  if (N < 128 || K < 128 || N % 128 != 0 || K % 128 != 0 || N > kMaxDim || K > kMaxDim ||
      N / 128 > 65535)
    return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(w) || !aligned16(q) || !aligned16(s) || !aligned16(q_t) || !aligned16(s_t))
    return FP8FG_ERR_MISALIGNED;
  if (!have_device()) return FP8FG_ERR_CUDA;
  return from_cuda(launch_weight_quant(w, w_dtype, N, K, q, s, q_t, s_t,
                                       (flags & FP8FG_POW2) != 0, as_stream(stream)));
}

namespace {

// Host checks shared by the dense GEMM entry points (no CUDA call).
fp8fg_status check_gemm_args(const uint8_t* a, const float* sa, const uint8_t* b, const float* sb,
                             void* c, fp8fg_dtype c_dtype, int64_t M, int64_t N, int64_t K,
                             unsigned flags, unsigned allowed) {
  if (!valid_dtype(c_dtype) || (flags & ~allowed) != 0 || M < 0 || N < 0 || K < 0)
    return FP8FG_ERR_INVALID_ARG;
  if ((flags & FP8FG_B_TILE1x128) && (flags & FP8FG_WHOLE_K)) return FP8FG_ERR_INVALID_ARG;
  if ((flags & FP8FG_STREAM_K) && (flags & FP8FG_WHOLE_K)) return FP8FG_ERR_INVALID_ARG;
  if (b == nullptr || sb == nullptr || (M > 0 && (a == nullptr || sa == nullptr || c == nullptr)))
    return FP8FG_ERR_INVALID_ARG;
  const bool b_tile = (flags & FP8FG_B_TILE1x128) != 0;
  if (K < 128 || K % 128 != 0 || N < 16 || (b_tile ? N % 16 != 0 : N % 128 != 0) || M > kMaxDim ||
      N > kMaxDim || K > kMaxDim)
    return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (((M + 127) / 128) * ((N + 255) / 256) > kMaxDim) return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(c))
    return FP8FG_ERR_MISALIGNED;
  return FP8FG_OK;
}

}  // namespace

fp8fg_status fp8_blockscaled_gemm(const uint8_t* a, const float* sa, const uint8_t* b,
                                  const float* sb, void* c, fp8fg_dtype c_dtype, int64_t M,
                                  int64_t N, int64_t K, unsigned flags, void* stream) {
  const fp8fg_status chk = check_gemm_args(a, sa, b, sb, c, c_dtype, M, N, K, flags,
                                           FP8FG_B_TILE1x128 | FP8FG_WHOLE_K);
  if (chk != FP8FG_OK) return chk;
  if (M == 0) return FP8FG_OK;
  if (!have_device()) return FP8FG_ERR_CUDA;
  return launch_gemm(a, sa, b, sb, c, c_dtype, M, N, K, (flags & FP8FG_B_TILE1x128) != 0,
                     (flags & FP8FG_WHOLE_K) != 0, nullptr, 0, false, as_stream(stream));
}

size_t fp8_blockscaled_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, unsigned flags) {
  if (M <= 0 || N <= 0 || K < 128 || K % 128 != 0 || (flags & FP8FG_WHOLE_K) || !have_device())
    return 0;
  return gemm_workspace_bytes(M, N, K, false, (flags & FP8FG_STREAM_K) != 0);
}

fp8fg_status fp8_blockscaled_gemm_ws(const uint8_t* a, const float* sa, const uint8_t* b,
                                     const float* sb, void* c, fp8fg_dtype c_dtype, int64_t M,
                                     int64_t N, int64_t K, unsigned flags, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  const fp8fg_status chk = check_gemm_args(a, sa, b, sb, c, c_dtype, M, N, K, flags,
                                           FP8FG_B_TILE1x128 | FP8FG_STREAM_K);
  if (chk != FP8FG_OK) return chk;
  if (!aligned16(workspace)) return FP8FG_ERR_MISALIGNED;
  if ((flags & FP8FG_STREAM_K) && workspace == nullptr) return FP8FG_ERR_INVALID_ARG;
  if (M == 0) return FP8FG_OK;
  if (!have_device()) return FP8FG_ERR_CUDA;
  const bool force = (flags & FP8FG_STREAM_K) != 0;
  if (workspace != nullptr && workspace_bytes < gemm_workspace_bytes(M, N, K, false, force))
    return FP8FG_ERR_INVALID_ARG;
  return launch_gemm(a, sa, b, sb, c, c_dtype, M, N, K, (flags & FP8FG_B_TILE1x128) != 0, false,
                     workspace, workspace_bytes, force, as_stream(stream));
}

fp8fg_status fp8_blockscaled_gemm_noalloc(const uint8_t* a, const float* sa, const uint8_t* b,
                                          const float* sb, void* c, fp8fg_dtype c_dtype, int64_t M,
                                          int64_t N, int64_t K, unsigned flags, void* stream) {
  const fp8fg_status chk = check_gemm_args(a, sa, b, sb, c, c_dtype, M, N, K, flags,
                                           FP8FG_B_TILE1x128 | FP8FG_STREAM_K);
  if (chk != FP8FG_OK) return chk;
  if (M == 0) return FP8FG_OK;
  if (!have_device()) return FP8FG_ERR_CUDA;
  return launch_gemm_noalloc(a, sa, b, sb, c, c_dtype, M, N, K, (flags & FP8FG_B_TILE1x128) != 0,
                             (flags & FP8FG_STREAM_K) != 0, as_stream(stream));
}

fp8fg_status fp8_blockscaled_gemm_quant(const uint8_t* a, const float* sa, const uint8_t* b,
                                        const float* sb, uint8_t* q, float* s, int64_t M,
                                        int64_t N, int64_t K, unsigned flags, void* stream) {
  if ((flags & ~(FP8FG_B_TILE1x128 | FP8FG_POW2)) != 0 || M < 0 || N < 0 || K < 0)
    return FP8FG_ERR_INVALID_ARG;
  if (b == nullptr || sb == nullptr || (M > 0 && (a == nullptr || sa == nullptr || q == nullptr ||
                                                  s == nullptr)))
    return FP8FG_ERR_INVALID_ARG;
  const bool b_tile = (flags & FP8FG_B_TILE1x128) != 0;
  if (K < 128 || K % 128 != 0 || N < 128 || N % 128 != 0 || M > kMaxDim || N > kMaxDim ||
      K > kMaxDim)
    return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (((M + 127) / 128) * ((N + 255) / 256) > kMaxDim) return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(q) ||
      !aligned16(s))
    return FP8FG_ERR_MISALIGNED;
  if (M == 0) return FP8FG_OK;
  if (!have_device()) return FP8FG_ERR_CUDA;
  return launch_gemm_quant(a, sa, b, sb, q, s, M, N, K, b_tile, (flags & FP8FG_POW2) != 0,
                           as_stream(stream));
}

fp8fg_status fp8_grouped_gemm(const uint8_t* a, const float* sa, const int32_t* offsets, int32_t E,
                              int64_t total_rows, const uint8_t* b, const float* sb, void* c,
                              fp8fg_dtype c_dtype, int64_t N, int64_t K, unsigned flags,
                              void* stream) {
  if (!valid_dtype(c_dtype) || flags != 0 || total_rows < 0 || N < 0 || K < 0 || E < 1)
    return FP8FG_ERR_INVALID_ARG;
  if (offsets == nullptr || b == nullptr || sb == nullptr ||
      (total_rows > 0 && (a == nullptr || sa == nullptr || c == nullptr)))
    return FP8FG_ERR_INVALID_ARG;
  if (E > 1024 || K < 128 || K % 128 != 0 || N < 128 || N % 128 != 0 || total_rows > kMaxDim ||
      N > kMaxDim || K > kMaxDim || static_cast<int64_t>(E) * N > kMaxDim ||
      (total_rows / 128 + E) * ((N + 255) / 256) > kMaxDim)
    return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(c) ||
      (reinterpret_cast<uintptr_t>(offsets) & 3u) != 0)
    return FP8FG_ERR_MISALIGNED;
  if (total_rows == 0) return FP8FG_OK;    // no rows: nothing to compute or write
  if (!have_device()) return FP8FG_ERR_CUDA;
  return launch_grouped_gemm(a, sa, offsets, E, total_rows, b, sb, c, c_dtype, N, K,
                             as_stream(stream));
}

fp8fg_status fp8_grouped_gemm_swiglu_quant(const uint8_t* a, const float* sa,
                                           const int32_t* offsets, int32_t E, int64_t total_rows,
                                           const uint8_t* b, const float* sb, uint8_t* q, float* s,
                                           int64_t N, int64_t K, unsigned flags, void* stream) {
  if ((flags & ~FP8FG_POW2) != 0 || total_rows < 0 || N < 0 || K < 0 || E < 1)
    return FP8FG_ERR_INVALID_ARG;
  if (offsets == nullptr || b == nullptr || sb == nullptr ||
      (total_rows > 0 && (a == nullptr || sa == nullptr || q == nullptr || s == nullptr)))
    return FP8FG_ERR_INVALID_ARG;
  if (E > 1024 || K < 128 || K % 128 != 0 || N < 256 || N % 256 != 0 || total_rows > kMaxDim ||
      N > kMaxDim || K > kMaxDim || static_cast<int64_t>(E) * N > kMaxDim ||
      (total_rows / 128 + E) * (N / 256) > kMaxDim)
    return FP8FG_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(sa) || !aligned16(b) || !aligned16(sb) || !aligned16(q) ||
      !aligned16(s) || (reinterpret_cast<uintptr_t>(offsets) & 3u) != 0)
    return FP8FG_ERR_MISALIGNED;
  if (total_rows == 0) return FP8FG_OK;    // no rows: nothing to compute or write
  if (!have_device()) return FP8FG_ERR_CUDA;
  return launch_grouped_swiglu_quant(a, sa, offsets, E, total_rows, b, sb, q, s, N, K,
                                     (flags & FP8FG_POW2) != 0, as_stream(stream));
}

fp8fg_status fp8_get_device_status(void* stream) {
  if (!have_device()) return FP8FG_ERR_CUDA;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return FP8FG_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return FP8FG_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess)
    return FP8FG_ERR_CUDA;
  return static_cast<fp8fg_status>(v);
}

fp8fg_status fp8fg_selftest_wait_timeout(uint32_t limit_cycles, void* stream) {
  if (limit_cycles == 0 || limit_cycles > (1u << 31)) return FP8FG_ERR_INVALID_ARG;
  if (!have_device()) return FP8FG_ERR_CUDA;
  return from_cuda(launch_wait_timeout_selftest(limit_cycles, as_stream(stream)));
}

}  // extern "C"
