// Host entry of the fused RMSNorm -> MXFP4 activation producer (norm_quant.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace mx {

struct NormQuantProblem {
  const void* x;        // bf16 [M][ldx]
  int ldx;
  void* residual;       // bf16 [M][ldr], updated in place to bf16(x + residual); or null
  int ldr;
  const void* gamma;    // bf16 [K]
  float eps;
  int M, K;
  uint8_t* codes;       // row-major [M][K/2] or the TILED codes region
  uint8_t* scales;      // row-major [M][ceil(K/32)] or the TILED scales region
  bool tiled;
  void* y;              // bf16 [M][ldy] normalized values that were quantized; or null
  int ldy;
};

cudaError_t launch_rmsnorm_quant(const NormQuantProblem& p, const DeviceInfo& dev, cudaStream_t s);
uint32_t norm_read_clear_error();
// Bound of the bulk-copy producer kernel's waits on its row copies, in SM
// clock cycles, for launches that follow (0 restores the default).
void set_norm_wait_cycles(long long cycles);

}  // namespace mx
