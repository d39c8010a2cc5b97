// Host-side declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mx {

// Tile geometry of the TILED layout (see include/mxfp4.h).
constexpr int kRowTile = 128;   // rows per tile / scale atom
constexpr int kKTile = 256;     // elements per tile along K (128 bytes of codes)
constexpr int kTileBytes = kRowTile * kKTile / 2;   // 16384
constexpr int kAtomBytes = 512;                     // 128 rows x 4 scales

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t padded_rows(int64_t R) { return ceil_div(R, kRowTile) * kRowTile; }
inline int64_t padded_k(int64_t K) { return ceil_div(K, kKTile) * kKTile; }
inline int64_t tiled_code_bytes(int64_t R, int64_t K) { return padded_rows(R) * padded_k(K) / 2; }
inline int64_t tiled_scale_bytes(int64_t R, int64_t K) { return padded_rows(R) * padded_k(K) / 32; }

// Packed weights (see include/mxfp4.h): one block per (256-row pair, k-tile)
// holding the pair's two code tiles and four scale atoms.
constexpr int kPairRows = 256;
constexpr int kWeightBlockBytes = 2 * kTileBytes + 4 * kAtomBytes;   // 34816
inline int64_t weight_rows(int64_t R) { return ceil_div(R, kPairRows) * kPairRows; }
inline int64_t weight_packed_bytes(int64_t R, int64_t K) {
  return weight_rows(R) / kPairRows * (padded_k(K) / kKTile) * kWeightBlockBytes;
}

// Error bits recorded in a translation unit's device error word.
constexpr uint32_t kErrTimeout = 1u;

// Largest stream-K grid the decode GEMM uses; sizes its partial-sum slots.
constexpr int kMaxStreamKCtas = 256;
// Largest activation row count served by the decode kernel.
constexpr int kDecodeMaxM = 64;
// Largest activation row count the decode kernel quantizes itself (each CTA
// its own k-steps, every quantizing warp one row); above it the standalone
// quantizer runs first and the kernel copies the quantized rows in.
constexpr int kDecodeLocalQuantMaxM = 8;

// Activation rows of a 128-row tile the GEMM loads: 16, 32 or 64 when
// M <= kDecodeMaxM (only those rows of the tiled activations are read), else 128.
inline int gemm_rows_a(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128)); }

struct DeviceInfo {
  int device;
  int sm_count;
  bool ok;   // an sm_103 device
};
// Properties of the current device, cached per device.
cudaError_t current_device_info(DeviceInfo* out);

// quant.cu
// Output layout of the activation quantizer: row-major, TILED (public), or
// blocked (the library's own workspace form: per (row tile, k-tile) the code
// rows followed by the two scale atoms, one bulk copy per GEMM stage).
enum class ActLayout { kRowMajor, kTiled, kBlocked };
inline int64_t blocked_bytes(int64_t M, int64_t K, int block_rows) {
  return ceil_div(M, kRowTile) * (padded_k(K) / kKTile) * (static_cast<int64_t>(block_rows) * 128 + 1024);
}
// rows: kTiled: rows of the tiled output to write (0 = all Rp rows);
// kBlocked: rows per block (128 for any M; 16/32/64 when M <= that).
cudaError_t launch_quant(const void* x, int M, int K, int ldx, uint8_t* codes, uint8_t* scales, ActLayout layout,
                         int rows, const DeviceInfo& dev, cudaStream_t s);
// Row-major codes/scales -> TILED activation layout (codes region, then scales).
cudaError_t launch_pack(const uint8_t* codes, const uint8_t* scales, int batch, int R, int K, uint8_t* packed,
                        const DeviceInfo& dev, cudaStream_t s);
// Row-major codes/scales -> packed weight blocks.
cudaError_t launch_pack_weights(const uint8_t* codes, const uint8_t* scales, int batch, int N, int K,
                                uint8_t* packed, const DeviceInfo& dev, cudaStream_t s);
// An empty ordinary launch: programmatic dependents launched after it start
// only once every earlier kernel on the stream has completed.
cudaError_t launch_ordering(const DeviceInfo& dev, cudaStream_t s);
uint32_t quant_read_clear_error();

// gemm.cu
struct GemmProblem {
  const uint8_t* a_codes;   // TILED activation codes, or the blocked activations (a_blocked)
  const uint8_t* a_scales;  // TILED activation scales (unused when a_blocked)
  bool a_blocked;           // a_codes holds blocked activations with 128-row blocks
  const uint8_t* w_packed;  // packed weights (codes region then scales region)
  const void* bias;         // bf16 [N] or null
  void* out;                // bf16 [M][ldo]; unused with MXFP4 output
  int ldo, M, N, K;
  uint8_t* qcodes;          // MXFP4 output (row-major codes [M][N/2], scales [M][ceil(N/32)]) or null
  uint8_t* qscales;
  bool splitcat;            // split + cat output (see OutView) instead of `out`
  void* cat;                // bf16 [M][H][s1 + s3]
  void* split;              // bf16 [M][H][s2]
  const void* z;            // bf16 [M][H][s3]
  int s1, s2, s3;
  void* workspace;          // stream-K partial sums
  size_t workspace_bytes;
  bool cta_pairs;           // the CTA-pair kernel (a diagnostic), or cudaErrorNotSupported where it does not apply
};
// Stream-K CTAs of the GEMM on this device, and the partial-sum + ticket
// workspace it needs for that grid.
int gemm_grid(const DeviceInfo& dev);
size_t gemm_streamk_workspace_bytes(int M, int N, int K, int grid);
cudaError_t launch_gemm(const GemmProblem& p, const DeviceInfo& dev, cudaStream_t s);
// CTA pairs the pair kernel runs an M x N problem on, or 0 where it does not
// apply (M <= kDecodeMaxM, an odd count of 128-row activation tiles below
// 16, or a last wave of 256 x 256 tiles more than 8% idle).
int gemm_pair_count(int M, int N, const DeviceInfo& dev);
uint32_t gemm_read_clear_error();

// decode.cu: M <= kDecodeMaxM in one launch.
struct DecodeProblem {
  const void* x;            // bf16 activations [M][ldx] (quantized by the kernel); null when a_codes/a_scales hold them
  int ldx;
  const uint8_t* a_codes;   // x == null: TILED activation codes, or the blocked activations (a_blocked)
  const uint8_t* a_scales;  // x == null: TILED activation scales (unused when a_blocked)
  bool a_blocked;           // a_codes holds blocked activations with gemm_rows_a(M)-row blocks
  const uint8_t* w_packed;
  const void* bias;
  void* out;
  int ldo, M, N, K;
  uint8_t* qcodes;          // MXFP4 output or null (as GemmProblem)
  uint8_t* qscales;
  bool splitcat;            // split + cat output (as GemmProblem)
  void* cat;
  void* split;
  const void* z;
  int s1, s2, s3;
};
cudaError_t launch_decode(const DecodeProblem& p, const DeviceInfo& dev, cudaStream_t s);
uint32_t decode_read_clear_error();
// Timeline stamps of the last decode launches (timeline build only): copies
// the stamp buffer to `host` and returns its element count, 0 in the default
// build, -1 on a CUDA error; *next_call = slot of the next launch.
int decode_stamps(unsigned long long* host, int* next_call);

// bmm.cu
cudaError_t launch_bmm(const void* x, const uint8_t* w_packed, void* out, int B, int M, int N, int K,
                       bool batch_major, const DeviceInfo& dev, cudaStream_t s);
uint32_t bmm_read_clear_error();

}  // namespace mx
