// synth_dev.cu -- device twin of synth.c: the same seeded, counter-based
// synthetic input generator, writing straight into device memory so that
// workloads of tens to hundreds of GB never pass through the host.
//
// Harness code, not part of the product path.  It holds none of the method's
// arithmetic.  The definition (SplitMix64 counter draws, Irwin-Hall(12)
// normal, mu + sigma*z with single IEEE binary64 roundings, RN to binary32,
// RNE to bf16) is stated in synth.c; every binary64 step below uses the
// explicitly rounded intrinsics so that no multiply-add is fused and the
// result matches the host bit-for-bit.
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

struct Dist {
  double mu, sigma, outlier_p, outlier_scale;
  int absval;
};

__device__ inline double value_at(uint64_t key, uint64_t i, const Dist& d) {
  int64_t ksum = 0;
#pragma unroll
  for (uint64_t j = 0; j < 6; ++j) {
    uint64_t w = mix64(key + (8u * i + j + 1u) * kGamma);
    ksum += (int64_t)(w >> 32);
    ksum += (int64_t)(w & 0xFFFFFFFFull);
  }
  double z = __dmul_rn(__ll2double_rn(ksum + 6 - 6 * (int64_t)0x100000000ll), 0x1p-32);
  double x = __dadd_rn(d.mu, __dmul_rn(d.sigma, z));
  if (d.outlier_p > 0.0) {
    uint64_t w = mix64(key + (8u * i + 6u + 1u) * kGamma);
    double u = __dmul_rn(__ull2double_rn(w >> 11), 0x1p-53);
    if (u < d.outlier_p) x = __dmul_rn(x, d.outlier_scale);
  }
  if (d.absval && x < 0.0) x = -x;
  return x;
}

__device__ inline uint16_t bf16_rne_bits(float f) {
  uint32_t b = __float_as_uint(f);
  uint32_t up = b >> 16, low = b & 0xFFFFu;
  if (low > 0x8000u || (low == 0x8000u && (up & 1u))) up += 1u;
  return (uint16_t)up;
}

__global__ void fill_kernel(void* out, int kind, int64_t start, int64_t count,
                            uint64_t key, Dist d) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < count; k += stride) {
    float f = __double2float_rn(value_at(key, (uint64_t)(start + k), d));
    if (kind == 0) static_cast<uint16_t*>(out)[k] = bf16_rne_bits(f);
    else if (kind == 2) static_cast<uint16_t*>(out)[k] = __half_as_ushort(__float2half_rn(f));
    else static_cast<float*>(out)[k] = f;
  }
}

}  // namespace

// Fill `count` elements of device buffer `out` (bf16 when kind == 0, fp32
// when kind == 1, fp16 when kind == 2) with elements start .. start+count-1 of stream (seed,
// stream).  Returns a cudaError_t value (0 on success).  Asynchronous on
// `stream_handle` (a cudaStream_t).
extern "C" int syn_fill_device(void* out, int kind, int64_t start, int64_t count,
                               uint64_t seed, uint64_t stream, double mu, double sigma,
                               double outlier_p, double outlier_scale, int absval,
                               void* stream_handle) {
  if (count <= 0) return 0;
  if (out == nullptr || kind < 0 || kind > 2) return (int)cudaErrorInvalidValue;
  uint64_t key = mix64(seed * kGamma + mix64(stream + 0x632BE59BD9B4E019ull));
  Dist d{mu, sigma, outlier_p, outlier_scale, absval};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return (int)e;
  int64_t blocks = (count + 255) / 256;
  int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream_handle>>>(out, kind, start, count,
                                                                      key, d);
  return (int)cudaGetLastError();
}
