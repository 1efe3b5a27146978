// Device twin of the seeded input generator in synth/__init__.py:
// Philox4x32-10 (Salmon et al., SC'11) keyed per tensor, Irwin-Hall sums of
// four 16-bit uniforms, per-row (or per-64-element) absmax integer
// quantisation and int4 / int2 packing.
// Every step is integer arithmetic except one IEEE double multiply and one
// round-to-nearest conversion per scale, so it matches the numpy version bit
// for bit.  Holds none of the MoE layer's arithmetic.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ void philox(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c[0]), lo0 = 0xD2511F53u * c[0];
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]), lo1 = 0xCD9E8D57u * c[2];
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
  }
}

__device__ __forceinline__ void pair_normals(uint64_t call, uint32_t k0, uint32_t k1, int* z0, int* z1) {
  uint32_t c[4] = {(uint32_t)call, (uint32_t)(call >> 32), 0u, 0u};
  philox(c, k0, k1);
  *z0 = (int)((c[0] & 0xFFFFu) + (c[0] >> 16) + (c[1] & 0xFFFFu) + (c[1] >> 16)) - 131070;
  *z1 = (int)((c[2] & 0xFFFFu) + (c[2] >> 16) + (c[3] & 0xFFFFu) + (c[3] >> 16)) - 131070;
}

__device__ __forceinline__ int quant(int z, long long amax, int qmax) {
  if (amax == 0) return 0;
  const long long a = z < 0 ? -(long long)z : (long long)z;
  const long long q = (2LL * qmax * a + amax) / (2LL * amax);
  return z < 0 ? -(int)q : (int)q;
}

// One block per row (grid-stride): pass 1 row absmax, pass 2 codes.
__global__ void __launch_bounds__(256) quant_rows_kernel(uint32_t k0, uint32_t k1, int rows, int K, int qmax,
                                                         double c, int bits, uint8_t* __restrict__ out,
                                                         float* __restrict__ scales) {
  __shared__ int red[8];
  const int half = K / 2;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint64_t base = (uint64_t)row * (uint64_t)half;
    int m = 0;
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
      int z0, z1;
      pair_normals(base + j, k0, k1, &z0, &z1);
      m = max(m, max(abs(z0), abs(z1)));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    int amax = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = max(amax, red[w]);
    __syncthreads();
    if (bits == 2) {
      // one byte per four elements (two draws), codes clamped to [-2, 1]
      for (int j = threadIdx.x; j < K / 4; j += blockDim.x) {
        int z[4];
        pair_normals(base + 2 * j, k0, k1, &z[0], &z[1]);
        pair_normals(base + 2 * j + 1, k0, k1, &z[2], &z[3]);
        uint32_t b = 0;
#pragma unroll
        for (int m = 0; m < 4; ++m) b |= (uint32_t)(min(quant(z[m], amax, qmax), 1) + 2) << (2 * m);
        out[(size_t)row * (K / 4) + j] = (uint8_t)b;
      }
    } else {
      for (int j = threadIdx.x; j < half; j += blockDim.x) {
        int z0, z1;
        pair_normals(base + j, k0, k1, &z0, &z1);
        const int q0 = quant(z0, amax, qmax), q1 = quant(z1, amax, qmax);
        if (bits == 4) {
          out[(size_t)row * half + j] = (uint8_t)((q0 + 8) | ((q1 + 8) << 4));
        } else {
          out[(size_t)row * K + 2 * j] = (uint8_t)(int8_t)q0;
          out[(size_t)row * K + 2 * j + 1] = (uint8_t)(int8_t)q1;
        }
      }
    }
    if (threadIdx.x == 0) scales[row] = __double2float_rn((double)amax * c);
  }
}

// One warp per run of 64 elements of a row (32 draws, one per lane): the run's
// absmax, its codes and its scale (scales [rows][K/64], row-major).
__global__ void __launch_bounds__(256) quant_groups64_kernel(uint32_t k0, uint32_t k1, int rows, int K, int qmax,
                                                             double c, int bits, uint8_t* __restrict__ out,
                                                             float* __restrict__ scales) {
  const int half = K / 2, ng = K / 64, lane = threadIdx.x & 31;
  const long long nw = (long long)rows * ng;
  for (long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < nw;
       w += ((long long)gridDim.x * blockDim.x) >> 5) {
    const int row = (int)(w / ng), g = (int)(w % ng);
    const int j = g * 32 + lane;  // draw index within the row
    int z0, z1;
    pair_normals((uint64_t)row * (uint64_t)half + j, k0, k1, &z0, &z1);
    int m = max(abs(z0), abs(z1));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int q0 = quant(z0, m, qmax), q1 = quant(z1, m, qmax);
    if (bits == 4) {
      out[(size_t)row * half + j] = (uint8_t)((q0 + 8) | ((q1 + 8) << 4));
    } else {
      out[(size_t)row * K + 2 * j] = (uint8_t)(int8_t)q0;
      out[(size_t)row * K + 2 * j + 1] = (uint8_t)(int8_t)q1;
    }
    if (lane == 0) scales[(size_t)row * ng + g] = __double2float_rn((double)m * c);
  }
}

__global__ void normal_f32_kernel(uint32_t k0, uint32_t k1, long long n, float mul, float* __restrict__ out) {
  const long long pairs = (n + 1) / 2;
  for (long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x; j < pairs;
       j += (long long)gridDim.x * blockDim.x) {
    int z0, z1;
    pair_normals((uint64_t)j, k0, k1, &z0, &z1);
    out[2 * j] = __fmul_rn((float)z0, mul);
    if (2 * j + 1 < n) out[2 * j + 1] = __fmul_rn((float)z1, mul);
  }
}

}  // namespace

extern "C" {

// Quantised weight matrix [rows][K]: bytes (int4 / int2 packed or int8) and scales.
int synth_quant_rows(uint32_t k0, uint32_t k1, int rows, int K, int qmax, double c, int bits, void* out,
                     float* scales, cudaStream_t st) {
  if (K % 2 || rows <= 0 || (bits == 2 && K % 4)) return -1;
  int grid = rows < 4096 ? rows : 4096;
  quant_rows_kernel<<<grid, 256, 0, st>>>(k0, k1, rows, K, qmax, c, bits, static_cast<uint8_t*>(out), scales);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

// The same with one scale per 64 elements of a row (K a multiple of 64).
int synth_quant_groups64(uint32_t k0, uint32_t k1, int rows, int K, int qmax, double c, int bits, void* out,
                         float* scales, cudaStream_t st) {
  if (K % 64 || rows <= 0 || bits == 2) return -1;
  const long long warps = (long long)rows * (K / 64);
  const long long blocks = (warps + 7) / 8 < 65536 ? (warps + 7) / 8 : 65536;
  quant_groups64_kernel<<<(unsigned)blocks, 256, 0, st>>>(k0, k1, rows, K, qmax, c, bits, static_cast<uint8_t*>(out),
                                                          scales);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

int synth_normal_f32(uint32_t k0, uint32_t k1, long long n, float mul, float* out, cudaStream_t st) {
  if (n <= 0) return 0;
  long long blocks = ((n + 1) / 2 + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  normal_f32_kernel<<<(unsigned)blocks, 256, 0, st>>>(k0, k1, n, mul, out);
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // extern "C"
