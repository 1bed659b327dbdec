// kvgen.cu -- device side of the seeded workload generator.
//
// Fills device buffers with the same bits as the host generator in
// workload/__init__.py: value(key, i) = round16(fp32(S - 131070) * scale),
// S = sum of the four 16-bit fields of SplitMix64(key + (i + 1) * gamma)
// (Steele, Lea and Flood, OOPSLA 2014). `scale` is passed in by the host so
// that both sides multiply by the very same fp32 number. Input generation
// only: nothing of the KV-injection method is computed here.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t value_bits(uint64_t key, uint64_t idx, float scale, int dtype) {
  uint64_t h = mix64(key + (idx + 1ull) * 0x9E3779B97F4A7C15ull);
  int s = (int)(h & 0xFFFF) + (int)((h >> 16) & 0xFFFF) + (int)((h >> 32) & 0xFFFF) + (int)(h >> 48);
  float x = __fmul_rn((float)(s - 131070), scale);
  if (dtype == 1) return __half_as_ushort(__float2half_rn(x));
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__global__ void fill_linear_kernel(uint16_t *dst, int64_t n, uint64_t key, uint64_t start,
                                   float scale, int dtype) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x * 8;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < n; i += stride) {
    if (i + 8 <= n) {
      uint16_t v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = value_bits(key, start + (uint64_t)(i + k), scale, dtype);
      uint4 w;
      w.x = v[0] | ((uint32_t)v[1] << 16);
      w.y = v[2] | ((uint32_t)v[3] << 16);
      w.z = v[4] | ((uint32_t)v[5] << 16);
      w.w = v[6] | ((uint32_t)v[7] << 16);
      if ((reinterpret_cast<uintptr_t>(dst + i) & 15) == 0) {
        *reinterpret_cast<uint4 *>(dst + i) = w;
      } else {
        for (int k = 0; k < 8; ++k) dst[i + k] = v[k];
      }
    } else {
      for (int64_t k = i; k < n; ++k) dst[k] = value_bits(key, start + (uint64_t)k, scale, dtype);
    }
  }
}

__global__ void fill_rows_kernel(uint16_t *dst, int64_t n_rows, int64_t row_len,
                                 const int64_t *row_base, uint64_t key, float scale, int dtype) {
  int64_t n = n_rows * row_len;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    int64_t r = i / row_len, e = i - r * row_len;
    dst[i] = value_bits(key, (uint64_t)(row_base[r] + e), scale, dtype);
  }
}

int grid_for(int64_t work, int threads) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = (work + threads - 1) / threads;
  int64_t cap = (int64_t)sms * 16;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

extern "C" {

// dst[i] = value(key, start + i), i < n; dtype 0 = bf16, 1 = fp16. Returns a cudaError_t.
int kvgen_fill_linear(void *dst, int64_t n, uint64_t key, uint64_t start, float scale, int dtype,
                      cudaStream_t stream) {
  if (n <= 0) return 0;
  fill_linear_kernel<<<grid_for((n + 7) / 8, 256), 256, 0, stream>>>((uint16_t *)dst, n, key,
                                                                       start, scale, dtype);
  return (int)cudaGetLastError();
}

// dst[r][e] = value(key, row_base[r] + e), r < n_rows, e < row_len; row_base on the device.
int kvgen_fill_rows(void *dst, int64_t n_rows, int64_t row_len, const int64_t *row_base,
                    uint64_t key, float scale, int dtype, cudaStream_t stream) {
  if (n_rows <= 0 || row_len <= 0) return 0;
  fill_rows_kernel<<<grid_for(n_rows * row_len, 256), 256, 0, stream>>>(
      (uint16_t *)dst, n_rows, row_len, row_base, key, scale, dtype);
  return (int)cudaGetLastError();
}

}  // extern "C"
