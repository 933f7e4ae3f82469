// Seeded synthetic input generator shared by the CPU oracle's tests and the CUDA path's tests and bench.
//
// It holds none of the prune step's arithmetic: it only turns (seed, stream, index) into numbers.
// Every value is a pure function of its counter, so any row of a 30 GB cache can be regenerated on the
// host one row at a time, and the device fill writes bit-identical values.
//
// Definitions (all integer or exactly-representable float arithmetic, so host and device agree bit for bit):
//   mix64(z)          : the SplitMix64 output function (Steele, Lea & Flood, "Fast splittable pseudorandom
//                       number generators", OOPSLA 2014): z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
//                       z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31.
//   stream_key(s, k)  : mix64(mix64(s + G) ^ (k * 0xD1B54A32D192ED03)), G = 0x9E3779B97F4A7C15.
//   word(key, i)      : mix64(key + (i + 1) * G), i.e. the i-th output of a SplitMix64 sequence seeded at key.
//   normal(key, i)    : Irwin-Hall sum of twelve 16-bit uniforms taken from word(key, 3i..3i+2):
//                       (sum_r r_k - 393210) / 65536.  Mean 0, variance (1 - 2^-32), support [-6, 6].
//                       The value is an exact fp32 number.
//   uniform(key, i)   : (word(key, i) >> 11) * 2^-53, a double in [0, 1).
//   bf16(x)           : round-to-nearest-even of the fp32 value x to bfloat16 (exact integer bit arithmetic).
#include <stdint.h>
#include <string.h>
#include <cuda_runtime.h>

#include <thread>
#include <vector>

#define SY_HD __host__ __device__ __forceinline__

static constexpr uint64_t SY_GOLDEN = 0x9E3779B97F4A7C15ull;

SY_HD uint64_t sy_mix64(uint64_t z) {
  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27; z *= 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

SY_HD uint64_t sy_stream_key(uint64_t seed, uint64_t stream) {
  return sy_mix64(sy_mix64(seed + SY_GOLDEN) ^ (stream * 0xD1B54A32D192ED03ull));
}

SY_HD uint64_t sy_word(uint64_t key, uint64_t i) { return sy_mix64(key + (i + 1) * SY_GOLDEN); }

SY_HD float sy_normal(uint64_t key, uint64_t i) {
  int32_t acc = 0;
  for (int w = 0; w < 3; ++w) {
    uint64_t r = sy_word(key, 3 * i + (uint64_t)w);
    acc += (int32_t)(r & 0xFFFF) + (int32_t)((r >> 16) & 0xFFFF) + (int32_t)((r >> 32) & 0xFFFF) +
           (int32_t)(r >> 48);
  }
  return (float)(acc - 393210) * (1.0f / 65536.0f);  // both steps are exact
}

SY_HD uint16_t sy_bf16_rne(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + bias) >> 16);
}

// ------------------------------------------------------------------------------------------------ host API
extern "C" {

uint64_t synth_stream_key(uint64_t seed, uint64_t stream) { return sy_stream_key(seed, stream); }
uint64_t synth_word(uint64_t key, uint64_t i) { return sy_word(key, i); }

void synth_normal_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset) {
  uint64_t key = sy_stream_key(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = sy_normal(key, (uint64_t)(offset + i));
}

void synth_uniform_f64(double* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset) {
  uint64_t key = sy_stream_key(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = (double)(sy_word(key, (uint64_t)(offset + i)) >> 11) * 0x1.0p-53;
}

// Rows of a [planes][plane_rows][D] tensor. Row r of plane p (r in [row0, row0 + rows)) gets the values
// normal(key, ((p * rows_per_plane_key) + (r - row0 + key_row0)) * D + e), so a chunk's content does not depend on
// where in the cache it is placed. dtype 0 = bf16 (uint16 bits), 1 = fp32.
void synth_fill_rows_host(void* out, int dtype, int64_t planes, int64_t plane_stride_rows, int64_t row0, int64_t rows,
                          int64_t D, uint64_t seed, uint64_t stream, int64_t key_rows_per_plane, int64_t key_row0) {
  const uint64_t key = sy_stream_key(seed, stream);
  const int64_t total_rows = planes * rows;
  auto work = [&](int64_t r_begin, int64_t r_end) {
    for (int64_t pr = r_begin; pr < r_end; ++pr) {
      const int64_t p = pr / rows, r = pr % rows;
      for (int64_t e = 0; e < D; ++e) {
        const uint64_t ctr = (uint64_t)(((p * key_rows_per_plane) + key_row0 + r) * D + e);
        const float x = sy_normal(key, ctr);
        const int64_t at = (p * plane_stride_rows + row0 + r) * D + e;
        if (dtype == 0) ((uint16_t*)out)[at] = sy_bf16_rne(x);
        else ((float*)out)[at] = x;
      }
    }
  };
  // The values do not depend on how the rows are split between threads.
  int64_t nt = (int64_t)std::thread::hardware_concurrency();
  if (nt < 1) nt = 1;
  if (nt > 32) nt = 32;
  if (total_rows * D < (int64_t)1 << 16) nt = 1;
  std::vector<std::thread> pool;
  for (int64_t t = 1; t < nt; ++t)
    pool.emplace_back(work, total_rows * t / nt, total_rows * (t + 1) / nt);
  work(0, total_rows / nt);
  for (auto& th : pool) th.join();
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------ device fill
__global__ void sy_fill_rows_kernel(void* out, int dtype, int64_t planes, int64_t plane_stride_rows, int64_t row0,
                                    int64_t rows, int64_t D, uint64_t key, int64_t key_rows_per_plane,
                                    int64_t key_row0) {
  const int64_t total = planes * rows * D;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
    int64_t e = g % D;
    int64_t r = (g / D) % rows;
    int64_t p = g / (D * rows);
    uint64_t ctr = (uint64_t)(((p * key_rows_per_plane) + key_row0 + r) * D + e);
    float x = sy_normal(key, ctr);
    int64_t at = (p * plane_stride_rows + row0 + r) * D + e;
    if (dtype == 0) ((uint16_t*)out)[at] = sy_bf16_rne(x);
    else ((float*)out)[at] = x;
  }
}

extern "C" int synth_fill_rows_device(void* out, int dtype, int64_t planes, int64_t plane_stride_rows, int64_t row0,
                                      int64_t rows, int64_t D, uint64_t seed, uint64_t stream,
                                      int64_t key_rows_per_plane, int64_t key_row0, void* cuda_stream) {
  if (planes <= 0 || rows <= 0 || D <= 0) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  const int64_t total = planes * rows * D;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * 32) blocks = (int64_t)sms * 32;
  sy_fill_rows_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)cuda_stream>>>(
      out, dtype, planes, plane_stride_rows, row0, rows, D, sy_stream_key(seed, stream), key_rows_per_plane,
      key_row0);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
