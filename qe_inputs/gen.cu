// gen.cu -- the seeded input generator of qe_inputs on the GPU, bit-identical to the numpy one.
//
// Holds none of the cache method's arithmetic: it only fills K/V/Q tensors.  Definitions (see
// qe_inputs/__init__.py): SplitMix64 row keys chained over (seed, tensor, batch, layer, head,
// position-or-step); channel c of a row draws splitmix64(key + 3c + j), j = 0..2, and sums the
// twelve 16-bit fields (Irwin-Hall); value = float(scale * (S - 393210)) / 65536 (exact), rounded
// to bf16 to nearest even.  Queries may add the exact mean of the original keys of a drift window.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__host__ __device__ __forceinline__ unsigned long long sm64(unsigned long long x) {
  unsigned long long z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ unsigned long long row_key(unsigned long long seed, long long tensor, long long b,
                                                               long long layer, long long head, long long pos) {
  unsigned long long k = sm64(seed);
  k = sm64(k ^ (unsigned long long)tensor);
  k = sm64(k ^ (unsigned long long)b);
  k = sm64(k ^ (unsigned long long)layer);
  k = sm64(k ^ (unsigned long long)head);
  k = sm64(k ^ (unsigned long long)pos);
  return k;
}

__device__ __forceinline__ int centred_sum(unsigned long long key, int c) {
  const unsigned long long base = key + 3ull * (unsigned long long)c;
  int s = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const unsigned long long r = sm64(base + (unsigned long long)j);
    s += (int)(r & 0xFFFF) + (int)((r >> 16) & 0xFFFF) + (int)((r >> 32) & 0xFFFF) + (int)(r >> 48);
  }
  return s - 393210;
}

__device__ __forceinline__ uint16_t bf16_rne(float f) {
  const unsigned b = __float_as_uint(f);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

constexpr int T_K = 1, T_V = 2, T_Q = 3, T_DRIFT = 5;

// out [B][H][n][d]; scale_int [H][d] or null
__global__ void gen_rows_kernel(unsigned long long seed, int tensor, int B, int layer, int H, int pos0, int n, int d,
                                const int* __restrict__ scale_int, uint16_t* __restrict__ out) {
  const long long rows = (long long)B * H * n;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int t = (int)(row % n);
    const int h = (int)((row / n) % H);
    const int b = (int)(row / ((long long)n * H));
    const unsigned long long key = row_key(seed, tensor, b, layer, h, pos0 + t);
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      const int sc = scale_int ? scale_int[h * d + c] : 1;
      const float f = (float)(centred_sum(key, c) * sc) / 65536.0f;
      out[row * d + c] = bf16_rne(f);
    }
  }
}

// queries of decode step `step` (1-based): out [B][Hq][d]; drift adds the exact mean key of a
// window drawn per (b, layer, kv head, epoch); kscale [Hkv][d] is the keys' channel scale
__global__ void gen_queries_kernel(unsigned long long seed, int B, int layer, int Hq, int G, int step, int d,
                                   int drift_period, int prefill, int window, const int* __restrict__ kscale,
                                   uint16_t* __restrict__ out) {
  extern __shared__ double mu[];   // [d]
  const int b = blockIdx.x / (Hq / G);
  const int kvh = blockIdx.x % (Hq / G);
  if (drift_period > 0) {
    const int epoch = (step - 1) / drift_period;
    const int first = epoch * drift_period + 1;
    const long long p = (long long)prefill + first - 1;
    const long long n_complete = p / window;
    const unsigned long long r = sm64(row_key(seed, T_DRIFT, b, layer, kvh, epoch));
    const long long j = (long long)(r % (unsigned long long)n_complete);
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      double s = 0.0;
      for (int t = 0; t < window; ++t) {
        const unsigned long long key = row_key(seed, T_K, b, layer, kvh, j * window + t);
        const float f = (float)(centred_sum(key, c) * kscale[kvh * d + c]) / 65536.0f;
        const uint16_t kb = bf16_rne(f);
        s += (double)__uint_as_float((unsigned)kb << 16);   // exact: multiples of 2^-16 below 2^7
      }
      mu[c] = s / window;
    }
  } else {
    for (int c = threadIdx.x; c < d; c += blockDim.x) mu[c] = 0.0;
  }
  __syncthreads();
  for (int i = 0; i < G; ++i) {
    const int h = kvh * G + i;
    const unsigned long long key = row_key(seed, T_Q, b, layer, h, step);
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      const float z = (float)centred_sum(key, c) / 65536.0f;
      const float f = drift_period > 0 ? __double2float_rn(__dadd_rn((double)z, mu[c])) : z;
      out[((size_t)b * Hq + h) * d + c] = bf16_rne(f);
    }
  }
}

}  // namespace

extern "C" {

int qe_gen_rows(unsigned long long seed, int tensor, int B, int layer, int H, int pos0, int n, int d,
                const int* scale_int, uint16_t* out, void* stream) {
  const long long rows = (long long)B * H * n;
  long long grid = rows < 65536 ? rows : 65536;
  if (grid < 1) return 0;
  gen_rows_kernel<<<(int)grid, 128, 0, (cudaStream_t)stream>>>(seed, tensor, B, layer, H, pos0, n, d, scale_int, out);
  return (int)cudaGetLastError();
}

int qe_gen_queries(unsigned long long seed, int B, int layer, int Hq, int G, int step, int d, int drift_period,
                   int prefill, int window, const int* kscale, uint16_t* out, void* stream) {
  gen_queries_kernel<<<B * (Hq / G), 128, d * sizeof(double), (cudaStream_t)stream>>>(
      seed, B, layer, Hq, G, step, d, drift_period, prefill, window, kscale, out);
  return (int)cudaGetLastError();
}

}  // extern "C"
