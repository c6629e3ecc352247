// The tiled layout of block-scale arrays: the order in which the block-scaled tensor-core
// GEMMs read the scales, so that one stage's scales of 128 rows arrive as one contiguous
// copy instead of one 16-byte request per row.
//
// A scale array has `rows` rows of `cols` scale bytes (one byte per block of 32 MXFP8 or
// 16 NVFP4 elements along K, rows in the [rows, cols] order the quantize passes write).
// Its bytes group into 32-bit words, word w of a row holding bytes 4w .. 4w + 3.  The tiled
// array is a sequence of 512-byte atoms, atom (t, w) for row tile t = r / 128 and word w at
// atom index t * ceil(cols / 4) + w; inside an atom, the word of row 128 t + 32 c + l sits
// at byte 16 l + 4 c.  That is the order tcgen05.cp.32x128b.warpx4 reads a 32-row x 16-byte
// block from shared memory into tensor-memory columns, where the scale-factor operand of
// tcgen05.mma.kind::mxf8f6f4 / kind::mxf4nvf4 (block_scale) expects the word of row 32 c + l
// in lane l, column c (PTX ISA, tcgen05 "scale factor" matrix layout).  Rows past `rows`
// and bytes past `cols` in the last atoms are zero.
//
// Page: "Generalized Tensor Parallelism (GTP)" (Megatron-Core developer guide), §1.3: the
// MXFP8 / NVFP4 scales themselves; their order in memory is not the pages' subject.
#include <algorithm>

#include "device.h"
#include "sm100_ptx.cuh"

namespace {

constexpr int kThreads = 256;

// One thread per 32-bit word of the tiled array; consecutive threads write consecutive
// words, and the 4 bytes of a word come from one row.
__global__ void __launch_bounds__(kThreads) sf_tile_kernel(const uint8_t *__restrict__ sf, int64_t rows, int64_t cols,
                                                           int64_t words, int64_t total, uint32_t *__restrict__ out) {
  gtp::ptx::allow_dependents();
  gtp::ptx::wait_prior_grid();
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t atom = i >> 7;
    const int within = int(i & 127);  // word index inside the atom: 4 l + c
    const int l = within >> 2, c = within & 3;
    const int64_t t = atom / words, w = atom - t * words;
    const int64_t r = t * 128 + 32 * c + l;
    uint32_t v = 0;
    if (r < rows) {
      const uint8_t *row = sf + r * cols;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t col = 4 * w + j;
        if (col < cols) v |= uint32_t(row[col]) << (8 * j);
      }
    }
    out[i] = v;
  }
}

}  // namespace

extern "C" int64_t gtp_sf_tiled_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return -1;
  return (rows + 127) / 128 * ((cols + 3) / 4) * 512;
}

extern "C" gtp_status gtp_sf_tile(const uint8_t *sf, int64_t rows, int64_t cols, uint8_t *tiled, gtp_stream stream) {
  gtp::clear_error();
  if (rows < 0 || cols < 0) return gtp::fail(GTP_E_ARG, "negative size");
  if (rows > (int64_t(1) << 40) / (cols ? cols : 1)) return gtp::fail(GTP_E_SHAPE, "array too large");
  if (rows == 0 || cols == 0) return GTP_OK;
  if (!sf || !tiled) return gtp::fail(GTP_E_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(tiled) & 3u) return gtp::fail(GTP_E_ALIGN, "tiled must be 4-byte aligned");
  gtp::DeviceInfo dev;
  if (gtp_status s = gtp::require_sm103(&dev)) return s;
  const int64_t words = (cols + 3) / 4;
  const int64_t total = (rows + 127) / 128 * words * 128;
  const int64_t want = (total + kThreads - 1) / kThreads;
  const int grid = int(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(dev.sm_count) * 8)));
  return gtp::launch_overlapped(sf_tile_kernel, grid, kThreads, 0, gtp::as_stream(stream), "sf_tile", sf, rows, cols,
                                words, total, reinterpret_cast<uint32_t *>(tiled));
}
