// NVFP4 activation quantiser (bloomery issue #565, §4, #687: W4A4 runs
// with 4-bit activations): one thread per 16-element block.
#include "common.cuh"

namespace gdn {

template <bool F32>
__global__ void __launch_bounds__(256) quantize_kernel(const void *__restrict__ x, int rows, int cols, float ts,
                                                       uint8_t *__restrict__ codes,
                                                       uint8_t *__restrict__ scales,
                                                       int32_t *status, const int32_t *row_slot, int num_slots,
                                                       int sf_tiled) {
  pdl_wait();  // x may come from the preceding kernel
  pdl_launch_dependents();
  const int nb = cols >> 4;
  const long long total = (long long)rows * nb;
  const float inv6ts = inv6ts_of(ts);
  for (long long blk = blockIdx.x * (long long)blockDim.x + threadIdx.x; blk < total;
       blk += (long long)gridDim.x * blockDim.x) {
    const long long r = blk / nb, b = blk % nb;
    float v[16];
    const bool live = !row_slot || (row_slot[r] >= 0 && row_slot[r] < num_slots);
    if (!live) {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    } else if (F32) {
      const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(x) + r * cols + b * 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float4 q = p[i];
        v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
      }
    } else {
      const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + r * cols + b * 16);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint4 q = p[i];
        uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
          v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      }
    }
    uint32_t lo, hi, s;
    if (!quant_block16(v, ts, inv6ts, lo, hi, s)) flag_status(status, GDN_E_NONFINITE);
    *reinterpret_cast<uint2 *>(codes + r * (cols >> 1) + b * 8) = make_uint2(lo, hi);
    if (sf_tiled)
      scales[sf_tiled_offset((int)r, (int)b, nb)] = uint8_t(s);
    else
      scales[r * nb + b] = uint8_t(s);
  }
}

cudaError_t launch_quantize(const void *x, int x_is_f32, int rows, int cols, float ts, uint8_t *codes,
                            uint8_t *scales, int32_t *status, cudaStream_t stream, const int32_t *row_slot,
                            int num_slots, bool pdl, bool sf_tiled) {
  const long long total = (long long)rows * (cols / 16);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (x_is_f32)
    return cudaLaunchKernelEx(&cfg, quantize_kernel<true>, x, rows, cols, ts, codes, scales, status, row_slot, num_slots,
                              (int)sf_tiled);
  return cudaLaunchKernelEx(&cfg, quantize_kernel<false>, x, rows, cols, ts, codes, scales, status, row_slot, num_slots,
                            (int)sf_tiled);
}

__global__ void tile_scales_kernel(const uint8_t *src, int rows, int K, uint8_t *dst) {
  const int nb = K / 16;
  const int prow = (rows + 127) / 128 * 128;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < (size_t)prow * nb; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / nb), b = (int)(i % nb);
    dst[sf_tiled_offset(r, b, nb)] = r < rows ? src[(size_t)r * nb + b] : uint8_t(0);
  }
}

cudaError_t launch_tile_scales(const uint8_t *src, int rows, int K, uint8_t *dst, cudaStream_t stream) {
  tile_scales_kernel<<<304, 256, 0, stream>>>(src, rows, K, dst);
  return cudaGetLastError();
}

// Codes [rows][K/2] -> 16 KB tiles of 128 rows x 128 bytes (256 values),
// tile (mt, kt) at ((mt * K/256) + kt) * 16 KB, each already in the 128-byte
// swizzled order the MMA's shared-memory descriptor expects: row r's 16-byte
// chunk c sits at r * 128 + ((c ^ (r % 8)) * 16). Rows past the end are zero.
__global__ void swizzle_tiles_kernel(const uint8_t *src, int rows, int K, uint8_t *dst) {
  const int nkt = K / 256;
  const size_t nchunks = (size_t)(rows + 127) / 128 * nkt * 1024;  // 16-byte chunks
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nchunks; i += (size_t)gridDim.x * blockDim.x) {
    const size_t tile = i >> 10;
    const int within = (int)(i & 1023), r = within >> 3, pos = within & 7;
    const int mt = (int)(tile / nkt), kt = (int)(tile % nkt);
    const int row = mt * 128 + r, c = pos ^ (r & 7);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < rows) v = *reinterpret_cast<const uint4 *>(src + (size_t)row * (K / 2) + kt * 128 + c * 16);
    *reinterpret_cast<uint4 *>(dst + i * 16) = v;
  }
}

cudaError_t launch_swizzle_tiles(const uint8_t *src, int rows, int K, uint8_t *dst, cudaStream_t stream) {
  if (K % 256) return cudaErrorInvalidValue;
  swizzle_tiles_kernel<<<304, 256, 0, stream>>>(src, rows, K, dst);
  return cudaGetLastError();
}

}  // namespace gdn
