// C ABI of the library (declared in include/mxfp4.h): argument checks on
// the host, workspace carving, dispatch to the kernels of quant.cu, gemm.cu
// and bmm.cu.  No entry point allocates device memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "mxfp4.h"
#include "mxfp4_diag.h"
#include "internal.h"
#include "norm_quant.h"

namespace mx {

// Per-device properties, filled once under a lock; the flag is published
// with release order so that a thread that sees it set sees the entry.
static DeviceInfo g_dev_cache[64];
static std::atomic<bool> g_dev_cached[64];
static std::mutex g_dev_mutex;

cudaError_t current_device_info(DeviceInfo* out) {
  int d = -1;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 64) return cudaErrorInvalidDevice;
  if (!g_dev_cached[d].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_dev_cached[d].load(std::memory_order_relaxed)) {
      *out = g_dev_cache[d];
      return cudaSuccess;
    }
    DeviceInfo info{d, 0, false};
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, d)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d)) != cudaSuccess) return e;
    info.ok = (major == 10 && minor == 3);
    g_dev_cache[d] = info;
    g_dev_cached[d].store(true, std::memory_order_release);
  }
  *out = g_dev_cache[d];
  return cudaSuccess;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Device check shared by every compute entry point.
static mxfp4_status device_ready(DeviceInfo* dev) {
  cudaError_t e = current_device_info(dev);
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return MXFP4_ERR_NO_DEVICE;
  if (e != cudaSuccess) return MXFP4_ERR_CUDA;
  return dev->ok ? MXFP4_OK : MXFP4_ERR_NO_DEVICE;
}

static mxfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA; }

// Workspace carve-up of mxfp4_gemm: tiled (or blocked) activation codes,
// tiled scales, stream-K partial sums, each 1 KiB aligned.
struct GemmWorkspace {
  size_t codes_off, scales_off, streamk_off, total;
};
static GemmWorkspace gemm_workspace_layout(int M, int N, int K, int grid) {
  GemmWorkspace w{};
  w.codes_off = 0;
  w.scales_off = w.codes_off + round_up(static_cast<size_t>(tiled_code_bytes(M, K)), 1024);
  w.streamk_off = w.scales_off + round_up(static_cast<size_t>(tiled_scale_bytes(M, K)), 1024);
  w.total = w.streamk_off + round_up(gemm_streamk_workspace_bytes(M, N, K, grid), 1024);
  return w;
}

// Stream-K grid of the current device (the largest grid if none is usable).
static int current_gemm_grid() {
  DeviceInfo dev;
  if (current_device_info(&dev) == cudaSuccess && dev.ok) return gemm_grid(dev);
  cudaGetLastError();   // clear the error of a failed device query
  return kMaxStreamKCtas;
}

}  // namespace mx

using namespace mx;

extern "C" {

int mxfp4_abi_version(void) { return 3; }

const char* mxfp4_status_string(mxfp4_status s) {
  switch (s) {
    case MXFP4_OK: return "MXFP4_OK";
    case MXFP4_ERR_INVALID_ARG: return "MXFP4_ERR_INVALID_ARG";
    case MXFP4_ERR_UNSUPPORTED_SHAPE: return "MXFP4_ERR_UNSUPPORTED_SHAPE";
    case MXFP4_ERR_MISALIGNED: return "MXFP4_ERR_MISALIGNED";
    case MXFP4_ERR_WORKSPACE: return "MXFP4_ERR_WORKSPACE";
    case MXFP4_ERR_CUDA: return "MXFP4_ERR_CUDA";
    case MXFP4_ERR_TIMEOUT: return "MXFP4_ERR_TIMEOUT";
    case MXFP4_ERR_NO_DEVICE: return "MXFP4_ERR_NO_DEVICE";
  }
  return "MXFP4_ERR_UNKNOWN";
}

size_t mxfp4_packed_weight_bytes(int batch, int N, int K) {
  if (batch <= 0 || N <= 0 || K <= 0 || (K & 1)) return 0;
  return static_cast<size_t>(batch) * static_cast<size_t>(weight_packed_bytes(N, K));
}

mxfp4_status mxfp4_weights_updated(void* stream) {
  DeviceInfo dev;
  mxfp4_status st = device_ready(&dev);
  if (st != MXFP4_OK) return st;
  return from_cuda(launch_ordering(dev, static_cast<cudaStream_t>(stream)));
}

size_t mxfp4_act_code_bytes(int M, int K, mxfp4_layout layout) {
  if (M <= 0 || K <= 0 || (K & 1)) return 0;
  if (layout == MXFP4_LAYOUT_ROWMAJOR) return static_cast<size_t>(M) * (K / 2);
  if (layout == MXFP4_LAYOUT_TILED) return static_cast<size_t>(tiled_code_bytes(M, K));
  return 0;
}

size_t mxfp4_act_scale_bytes(int M, int K, mxfp4_layout layout) {
  if (M <= 0 || K <= 0 || (K & 1)) return 0;
  if (layout == MXFP4_LAYOUT_ROWMAJOR) return static_cast<size_t>(M) * static_cast<size_t>(ceil_div(K, 32));
  if (layout == MXFP4_LAYOUT_TILED) return static_cast<size_t>(tiled_scale_bytes(M, K));
  return 0;
}

mxfp4_status mxfp4_pack_weights(const uint8_t* w_codes, const uint8_t* w_scales, int batch, int N, int K,
                                void* packed, void* stream) {
  if (w_codes == nullptr || w_scales == nullptr || packed == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (batch <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_INVALID_ARG;
  if (K & 1) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(packed)) return MXFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  mxfp4_status st = device_ready(&dev);
  if (st != MXFP4_OK) return st;
  return from_cuda(launch_pack_weights(w_codes, w_scales, batch, N, K, static_cast<uint8_t*>(packed), dev,
                               static_cast<cudaStream_t>(stream)));
}

mxfp4_status mxfp4_quant_act(const void* x, int M, int K, int ldx, uint8_t* codes, uint8_t* scales,
                             mxfp4_layout layout, void* stream) {
  if (x == nullptr || codes == nullptr || scales == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0) return MXFP4_ERR_INVALID_ARG;
  if (layout != MXFP4_LAYOUT_ROWMAJOR && layout != MXFP4_LAYOUT_TILED) return MXFP4_ERR_INVALID_ARG;
  if ((K & 1) || ldx < K) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if ((reinterpret_cast<uintptr_t>(x) & 1) != 0) return MXFP4_ERR_MISALIGNED;
  if (layout == MXFP4_LAYOUT_TILED && (!aligned16(codes) || !aligned16(scales))) return MXFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  mxfp4_status st = device_ready(&dev);
  if (st != MXFP4_OK) return st;
  return from_cuda(launch_quant(x, M, K, ldx, codes, scales, layout == MXFP4_LAYOUT_TILED ? ActLayout::kTiled : ActLayout::kRowMajor, 0, dev,
                                static_cast<cudaStream_t>(stream)));
}

mxfp4_status mxfp4_rmsnorm_quant_act(const void* x, int ldx, void* residual, int ldr, const void* gamma, float eps,
                                     int M, int K, uint8_t* codes, uint8_t* scales, mxfp4_layout layout, void* y,
                                     int ldy, void* stream) {
  if (x == nullptr || gamma == nullptr || codes == nullptr || scales == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (M <= 0 || K <= 0 || !(eps >= 0.f)) return MXFP4_ERR_INVALID_ARG;
  if (layout != MXFP4_LAYOUT_ROWMAJOR && layout != MXFP4_LAYOUT_TILED) return MXFP4_ERR_INVALID_ARG;
  if ((K & 1) || ldx < K || (residual != nullptr && ldr < K) || (y != nullptr && ldy < K))
    return MXFP4_ERR_UNSUPPORTED_SHAPE;
  auto odd = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1) != 0; };
  if (odd(x) || odd(gamma) || (residual != nullptr && odd(residual)) || (y != nullptr && odd(y)))
    return MXFP4_ERR_MISALIGNED;
  if (layout == MXFP4_LAYOUT_TILED && (!aligned16(codes) || !aligned16(scales))) return MXFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  mxfp4_status st = device_ready(&dev);
  if (st != MXFP4_OK) return st;
  NormQuantProblem p{x, ldx, residual, ldr, gamma, eps, M, K, codes, scales, layout == MXFP4_LAYOUT_TILED, y, ldy};
  return from_cuda(launch_rmsnorm_quant(p, dev, static_cast<cudaStream_t>(stream)));
}

size_t mxfp4_gemm_workspace_bytes(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0 || (K & 1)) return 0;
  return gemm_workspace_layout(M, N, K, current_gemm_grid()).total;
}

// The split + cat output form of mxfp4_gemm_split_cat (on: selected).
struct SplitCat {
  bool on;
  void* cat;
  void* split;
  const void* z;
  int s1, s2, s3;
};

// The GEMM behind mxfp4_gemm (bf16 `out`), mxfp4_gemm_mxfp4_out (qcodes /
// qscales set, `out` unused) and mxfp4_gemm_split_cat (sc.on).
static mxfp4_status gemm_any(const void* a_bf16, int lda, const uint8_t* a_codes, const uint8_t* a_scales,
                             mxfp4_layout a_layout, const void* w_packed, const void* bias, void* out, int ldo,
                             uint8_t* qcodes, uint8_t* qscales, int M, int N, int K, void* workspace,
                             size_t workspace_bytes, void* stream, const SplitCat& sc = SplitCat{},
                             bool cta_pairs = false) {
  const bool quant_out = qcodes != nullptr || sc.on;   // no bf16 [M][ldo] output
  if (w_packed == nullptr || (!quant_out && out == nullptr) || (qcodes != nullptr && qscales == nullptr))
    return MXFP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_INVALID_ARG;
  if (qcodes != nullptr && (N & 1)) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  const bool from_bf16 = a_bf16 != nullptr;
  if (from_bf16 && (a_codes != nullptr || a_scales != nullptr)) return MXFP4_ERR_INVALID_ARG;
  if (!from_bf16 && (a_codes == nullptr || a_scales == nullptr)) return MXFP4_ERR_INVALID_ARG;
  if (!from_bf16 && a_layout != MXFP4_LAYOUT_ROWMAJOR && a_layout != MXFP4_LAYOUT_TILED)
    return MXFP4_ERR_INVALID_ARG;
  if ((K & 1) || (!quant_out && ldo < N) || (from_bf16 && lda < K)) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(w_packed) || (!quant_out && !aligned16(out)) ||
      (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1)))
    return MXFP4_ERR_MISALIGNED;
  if (from_bf16 && (reinterpret_cast<uintptr_t>(a_bf16) & 1)) return MXFP4_ERR_MISALIGNED;
  if (!from_bf16 && a_layout == MXFP4_LAYOUT_TILED && (!aligned16(a_codes) || !aligned16(a_scales)))
    return MXFP4_ERR_MISALIGNED;
  if (workspace == nullptr) return MXFP4_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MXFP4_ERR_MISALIGNED;
  // without a usable device, check against the largest grid's requirement
  if (workspace_bytes < gemm_workspace_layout(M, N, K, kMaxStreamKCtas).total) {
    DeviceInfo probe;
    if (current_device_info(&probe) != cudaSuccess || !probe.ok) {
      cudaGetLastError();
      return MXFP4_ERR_WORKSPACE;
    }
  }

  DeviceInfo dev;
  mxfp4_status st = device_ready(&dev);
  if (st != MXFP4_OK) return st;
  const GemmWorkspace wl = gemm_workspace_layout(M, N, K, gemm_grid(dev));
  if (workspace_bytes < wl.total) return MXFP4_ERR_WORKSPACE;
  if (cta_pairs && gemm_pair_count(M, N, dev) <= 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  if (M <= kDecodeMaxM) {
    DecodeProblem d{};
    d.w_packed = static_cast<const uint8_t*>(w_packed);
    d.bias = bias;
    d.out = out;
    d.ldo = ldo;
    d.M = M;
    d.N = N;
    d.K = K;
    d.qcodes = qcodes;
    d.qscales = qscales;
    d.splitcat = sc.on;
    d.cat = sc.cat;
    d.split = sc.split;
    d.z = sc.z;
    d.s1 = sc.s1;
    d.s2 = sc.s2;
    d.s3 = sc.s3;
    if (from_bf16 && M <= kDecodeLocalQuantMaxM) {
      d.x = a_bf16;   // quantized inside the GEMM kernel
      d.ldx = lda;
    } else if (from_bf16) {
      // quantized by the standalone quantizer first, into the blocked form
      cudaError_t e =
          launch_quant(a_bf16, M, K, lda, ws + wl.codes_off, nullptr, ActLayout::kBlocked, gemm_rows_a(M), dev, s);
      if (e != cudaSuccess) return MXFP4_ERR_CUDA;
      d.a_codes = ws + wl.codes_off;
      d.a_blocked = true;
    } else if (a_layout == MXFP4_LAYOUT_ROWMAJOR) {
      // the pages' pre-quantized (x_fp4, x_scales) input: re-lay out, pad scales with 0x7F
      cudaError_t e = launch_pack(a_codes, a_scales, 1, M, K, ws + wl.codes_off, dev, s);
      if (e != cudaSuccess) return MXFP4_ERR_CUDA;
      d.a_codes = ws + wl.codes_off;
      d.a_scales = ws + wl.codes_off + tiled_code_bytes(M, K);
    } else {
      d.a_codes = a_codes;
      d.a_scales = a_scales;
    }
    return from_cuda(launch_decode(d, dev, s));
  }

  GemmProblem p{};
  if (from_bf16) {
    // quantized into the workspace in the blocked form (one copy per stage)
    p.a_codes = ws + wl.codes_off;
    p.a_scales = nullptr;
    p.a_blocked = true;
    cudaError_t e = launch_quant(a_bf16, M, K, lda, ws + wl.codes_off, nullptr, ActLayout::kBlocked, kRowTile, dev, s);
    if (e != cudaSuccess) return MXFP4_ERR_CUDA;
  } else if (a_layout == MXFP4_LAYOUT_ROWMAJOR) {
    // the pages' pre-quantized (x_fp4, x_scales) input: re-lay out, pad scales with 0x7F
    cudaError_t e = launch_pack(a_codes, a_scales, 1, M, K, ws + wl.codes_off, dev, s);
    if (e != cudaSuccess) return MXFP4_ERR_CUDA;
    p.a_codes = ws + wl.codes_off;
    p.a_scales = ws + wl.codes_off + tiled_code_bytes(M, K);
  } else {
    p.a_codes = a_codes;
    p.a_scales = a_scales;
  }
  p.w_packed = static_cast<const uint8_t*>(w_packed);
  p.bias = bias;
  p.out = out;
  p.ldo = ldo;
  p.M = M;
  p.N = N;
  p.K = K;
  p.qcodes = qcodes;
  p.qscales = qscales;
  p.splitcat = sc.on;
  p.cat = sc.cat;
  p.split = sc.split;
  p.z = sc.z;
  p.s1 = sc.s1;
  p.s2 = sc.s2;
  p.s3 = sc.s3;
  p.workspace = ws + wl.streamk_off;
  p.workspace_bytes = wl.total - wl.streamk_off;
  p.cta_pairs = cta_pairs;
  return from_cuda(launch_gemm(p, dev, s));
}

mxfp4_status mxfp4_gemm(const void* a_bf16, int lda, const uint8_t* a_codes, const uint8_t* a_scales,
                        mxfp4_layout a_layout, const void* w_packed, const void* bias, void* out, int ldo, int M,
                        int N, int K, void* workspace, size_t workspace_bytes, void* stream) {
  return gemm_any(a_bf16, lda, a_codes, a_scales, a_layout, w_packed, bias, out, ldo, nullptr, nullptr, M, N, K,
                  workspace, workspace_bytes, stream);
}

mxfp4_status mxfp4_diag_gemm_pair(const void* a_bf16, int lda, const uint8_t* a_codes, const uint8_t* a_scales,
                                  mxfp4_layout a_layout, const void* w_packed, const void* bias, void* out, int ldo,
                                  int M, int N, int K, void* workspace, size_t workspace_bytes, void* stream) {
  return gemm_any(a_bf16, lda, a_codes, a_scales, a_layout, w_packed, bias, out, ldo, nullptr, nullptr, M, N, K,
                  workspace, workspace_bytes, stream, SplitCat{}, true);
}

mxfp4_status mxfp4_gemm_mxfp4_out(const void* a_bf16, int lda, const uint8_t* a_codes, const uint8_t* a_scales,
                                  mxfp4_layout a_layout, const void* w_packed, const void* bias, uint8_t* out_codes,
                                  uint8_t* out_scales, int M, int N, int K, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  if (out_codes == nullptr || out_scales == nullptr) return MXFP4_ERR_INVALID_ARG;
  return gemm_any(a_bf16, lda, a_codes, a_scales, a_layout, w_packed, bias, nullptr, 0, out_codes, out_scales, M, N,
                  K, workspace, workspace_bytes, stream);
}

mxfp4_status mxfp4_gemm_split_cat(const void* a_bf16, int lda, const uint8_t* a_codes, const uint8_t* a_scales,
                                  mxfp4_layout a_layout, const void* w_packed, const void* bias, int M, int N, int K,
                                  int s1, int s2, const void* z, int s3, void* out_cat, void* out_split,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (s1 < 0 || s2 < 0 || s3 < 0 || s1 + s2 == 0) return MXFP4_ERR_INVALID_ARG;
  if ((s1 + s3 > 0 && out_cat == nullptr) || (s2 > 0 && out_split == nullptr) || (s3 > 0 && z == nullptr))
    return MXFP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0) return MXFP4_ERR_INVALID_ARG;
  if ((s1 % 8) || (s2 % 8) || (s3 % 8) || N % (s1 + s2) != 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if ((s1 + s3 > 0 && !aligned16(out_cat)) || (s2 > 0 && !aligned16(out_split)) || (s3 > 0 && !aligned16(z)))
    return MXFP4_ERR_MISALIGNED;
  SplitCat sc{true, out_cat, out_split, z, s1, s2, s3};
  return gemm_any(a_bf16, lda, a_codes, a_scales, a_layout, w_packed, bias, nullptr, 0, nullptr, nullptr, M, N, K,
                  workspace, workspace_bytes, stream, sc);
}

mxfp4_status a16wfp4_bmm(const void* x, const void* w_packed, void* out, int B, int M, int N, int K,
                         mxfp4_bmm_out_layout out_layout, void* stream) {
  if (x == nullptr || w_packed == nullptr || out == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (B <= 0 || M <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_INVALID_ARG;
  if (out_layout != MXFP4_OUT_BMN && out_layout != MXFP4_OUT_MBN) return MXFP4_ERR_INVALID_ARG;
  if (K % 64 != 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w_packed) || !aligned16(out)) return MXFP4_ERR_MISALIGNED;
  DeviceInfo dev;
  mxfp4_status st = device_ready(&dev);
  if (st != MXFP4_OK) return st;
  return from_cuda(launch_bmm(x, static_cast<const uint8_t*>(w_packed), out, B, M, N, K,
                              out_layout == MXFP4_OUT_MBN, dev, static_cast<cudaStream_t>(stream)));
}

mxfp4_status mxfp4_diag_set_wait_cycles(long long cycles) {
  if (cycles < 0) return MXFP4_ERR_INVALID_ARG;
  set_norm_wait_cycles(cycles);
  return MXFP4_OK;
}

mxfp4_status mxfp4_diag_decode_timeline(unsigned long long* host, size_t host_bytes, int* next_call) {
  if (host == nullptr || next_call == nullptr || host_bytes < 64u * 256u * 8u * sizeof(unsigned long long))
    return MXFP4_ERR_INVALID_ARG;
  const int n = decode_stamps(host, next_call);
  if (n == 0) return MXFP4_ERR_INVALID_ARG;   // the default build carries no stamps
  return n > 0 ? MXFP4_OK : MXFP4_ERR_CUDA;
}

mxfp4_status mxfp4_get_device_error(void* stream) {
  DeviceInfo dev;
  mxfp4_status st = device_ready(&dev);
  if (st != MXFP4_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MXFP4_ERR_CUDA;
  const uint32_t err = quant_read_clear_error() | gemm_read_clear_error() | decode_read_clear_error() |
                       bmm_read_clear_error() | norm_read_clear_error();
  return (err & kErrTimeout) ? MXFP4_ERR_TIMEOUT : MXFP4_OK;
}

}  // extern "C"
