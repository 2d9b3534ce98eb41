// Device implementation of the seeded input generator (see synth.h): the same
// SplitMix64 streams and Irwin-Hall(12) normals as synth_host.c, written on the GPU so
// that a 60 GB model never has to exist in host memory. Not part of the decode path.
#include <cuda_runtime.h>
#include <stdint.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

__device__ __forceinline__ uint64_t d_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}
__device__ __forceinline__ uint64_t d_splitmix(uint64_t x) { return d_mix64(x + GOLDEN); }
__host__ __device__ __forceinline__ uint64_t tid_of(int kind, int layer, int sub) {
  return ((uint64_t)(uint32_t)kind << 32) | ((uint64_t)(uint16_t)layer << 16) | (uint64_t)(uint16_t)sub;
}
static uint64_t h_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}
static uint64_t h_key(uint64_t seed, uint64_t tid) {
  return h_mix64((h_mix64(seed + GOLDEN) ^ tid) + GOLDEN);
}
__device__ __forceinline__ uint32_t d_sum16(uint64_t r) {
  return (uint32_t)(r & 0xFFFF) + (uint32_t)((r >> 16) & 0xFFFF) + (uint32_t)((r >> 32) & 0xFFFF) +
         (uint32_t)(r >> 48);
}
__device__ __forceinline__ float d_normal(uint64_t key, uint64_t i) {
  uint32_t s = d_sum16(d_splitmix(key + (3 * i) * GOLDEN)) + d_sum16(d_splitmix(key + (3 * i + 1) * GOLDEN)) +
               d_sum16(d_splitmix(key + (3 * i + 2) * GOLDEN));
  return __fmul_rn((float)((int32_t)s - 393216), 1.0f / 65536.0f);
}
__device__ __forceinline__ uint16_t d_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
__device__ __forceinline__ uint16_t d_value(uint64_t key, uint64_t i, float sigma, float offset, bool with_offset) {
  float v = __fmul_rn(sigma, d_normal(key, i));
  if (with_offset) v = __fadd_rn(offset, v);
  return d_bf16(v);
}

__global__ void fill_slice_kernel(uint64_t key, uint64_t start, uint64_t count, float sigma, float offset,
                                  int with_offset, uint16_t* out) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    out[i] = d_value(key, start + i, sigma, offset, with_offset != 0);
}

// Logical KV stream (layer, b, g) element pos*d+i written into the paged pool
// [L][num_pages][n_kv][page][d] at page block_table[b][pos / page].
__global__ void fill_kv_kernel(const uint64_t* keys /*[L][B][nkv]*/, int L, int B, int nkv, int d, int page,
                               const int32_t* ctx_len, const int32_t* block_table, int max_pages,
                               int64_t num_pages, uint16_t* pool) {
  const int lb = blockIdx.y, l = lb / B, b = lb % B;
  const int64_t n = (int64_t)ctx_len[b] * nkv * d;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
    const int i = (int)(e % d);
    const int g = (int)((e / d) % nkv);
    const int64_t pos = e / ((int64_t)d * nkv);
    const int pg = block_table[(int64_t)b * max_pages + pos / page];
    if (pg < 0 || pg >= num_pages) continue;
    const uint64_t key = keys[((int64_t)l * B + b) * nkv + g];
    const int64_t dst = ((((int64_t)l * num_pages + pg) * nkv + g) * page + pos % page) * d + i;
    pool[dst] = d_value(key, (uint64_t)pos * d + i, 1.0f, 0.0f, false);
  }
}

extern "C" {

// Fill [n_layer][n_sub][inner] bf16 with streams tid(kind, layer0 + l, s). Returns a cudaError_t.
int synth_dev_fill_stack(uint64_t seed, int kind, int layer0, int n_layer, int n_sub, uint64_t inner, float sigma,
                         float offset, void* out, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  uint16_t* o = (uint16_t*)out;
  for (int l = 0; l < n_layer; ++l)
    for (int s = 0; s < n_sub; ++s) {
      const uint64_t key = h_key(seed, tid_of(kind, layer0 + l, s));
      uint64_t blocks = (inner + 255) / 256;
      if (blocks > 8192) blocks = 8192;
      fill_slice_kernel<<<(unsigned)blocks, 256, 0, st>>>(key, 0, inner, sigma, offset, offset != 0.0f,
                                                          o + ((uint64_t)l * n_sub + s) * inner);
    }
  return (int)cudaGetLastError();
}

// Paged KV pool for `kind` (SYNTH_K or SYNTH_V). ctx_len and block_table are device arrays.
int synth_dev_fill_kv(uint64_t seed, int kind, int L, int B, int nkv, int d, int page, const int32_t* ctx_len,
                      int max_ctx, const int32_t* block_table, int max_pages, int64_t num_pages, void* pool,
                      void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  const size_t nkeys = (size_t)L * B * nkv;
  uint64_t* hkeys = new uint64_t[nkeys];
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < B; ++b)
      for (int g = 0; g < nkv; ++g) hkeys[((size_t)l * B + b) * nkv + g] = h_key(seed, tid_of(kind, l, b * nkv + g));
  uint64_t* dkeys = nullptr;
  cudaError_t e = cudaMallocAsync((void**)&dkeys, nkeys * sizeof(uint64_t), st);
  if (e != cudaSuccess) { delete[] hkeys; return (int)e; }
  cudaMemcpyAsync(dkeys, hkeys, nkeys * sizeof(uint64_t), cudaMemcpyHostToDevice, st);
  int64_t per = (int64_t)max_ctx * nkv * d;
  int64_t bx = (per + 255) / 256;
  if (bx > 2048) bx = 2048;
  if (bx < 1) bx = 1;
  dim3 grid((unsigned)bx, (unsigned)(L * B));
  fill_kv_kernel<<<grid, 256, 0, st>>>(dkeys, L, B, nkv, d, page, ctx_len, block_table, max_pages, num_pages,
                                       (uint16_t*)pool);
  e = cudaGetLastError();
  cudaStreamSynchronize(st);
  cudaFreeAsync(dkeys, st);
  cudaStreamSynchronize(st);
  delete[] hkeys;
  return (int)e;
}

}  // extern "C"
