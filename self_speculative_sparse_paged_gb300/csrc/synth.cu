// Device-side seeded synthetic K/V generator (input synthesis, not the method).
// Implements the same counter-based definition as the host generator
// (SplitMix64 draws, Irwin-Hall(4) normals, planted heavy-hitter keys,
// bf16 round-to-nearest-even); every floating-point step is one correctly
// rounded operation (__fmul_rn / __fadd_rn), so both sides agree bit for bit.
#include <cuda_bf16.h>

#include "kernels.h"

namespace vegas {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1ull) * kGolden);
}

// float32(sqrt(3) / 65536)
__device__ __forceinline__ float irwin_hall_normal(uint64_t r) {
  const int s = int(r & 0xFFFFull) + int((r >> 16) & 0xFFFFull) + int((r >> 32) & 0xFFFFull) +
                int(r >> 48) - 131070;
  return __fmul_rn(float(s), __uint_as_float(0x37ddb3d7u));
}

__device__ __forceinline__ uint16_t bf16_rne_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return uint16_t((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

struct SynthParams {
  uint16_t* cache;
  const int32_t* owner;
  const int32_t* ctx_lens;
  const int32_t* positions;
  const float* unit_dir;
  uint64_t key_val;     // K or V value stream key
  uint64_t key_heavy;   // heavy-position stream key
  uint64_t heavy_threshold;
  int heavy_last;
  int is_k;
  int num_pages, hkv, head_dim, max_pages;
};

__global__ void synth_kv_kernel(const SynthParams p) {
  const int d = p.head_dim;
  const size_t chunks = size_t(p.num_pages) * p.hkv * 16 * (d / 8);
  for (size_t c = blockIdx.x * size_t(blockDim.x) + threadIdx.x; c < chunks;
       c += size_t(gridDim.x) * blockDim.x) {
    const size_t e0 = c * 8;
    const int j0 = int(e0 % d);
    const size_t row = e0 / d;                 // (page * hkv + g) * 16 + slot
    const int slot = int(row % 16);
    const int g = int((row / 16) % p.hkv);
    const int page = int(row / (16 * size_t(p.hkv)));
    uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int own = p.owner[page];
    if (own >= 0) {
      const int b = own / p.max_pages;
      const int pos = (own % p.max_pages) * 16 + slot;
      if (pos < p.positions[b]) {
        const int L = p.ctx_lens[b];
        const uint64_t unit = uint64_t(b) * p.hkv + g;
        const uint64_t ctr_row = (unit << 24) + uint64_t(pos);
        bool heavy = false;
        if (p.is_k && pos < L)
          heavy = draw(p.key_heavy, ctr_row) < p.heavy_threshold || pos >= L - p.heavy_last;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int j = j0 + i;
          float z = irwin_hall_normal(draw(p.key_val, ctr_row * uint64_t(d) + uint64_t(j)));
          if (heavy) z = __fadd_rn(__fmul_rn(3.0f, p.unit_dir[j]), __fmul_rn(0.3f, z));
          v[i] = bf16_rne_bits(z);
        }
      }
    }
    uint4 w;
    w.x = uint32_t(v[0]) | (uint32_t(v[1]) << 16);
    w.y = uint32_t(v[2]) | (uint32_t(v[3]) << 16);
    w.z = uint32_t(v[4]) | (uint32_t(v[5]) << 16);
    w.w = uint32_t(v[6]) | (uint32_t(v[7]) << 16);
    *reinterpret_cast<uint4*>(p.cache + e0) = w;
  }
}

static uint64_t stream_key(uint64_t seed, uint64_t tag) { return mix64(seed + tag * kGolden); }

cudaError_t launch_synth_kv(void* cache, int which, uint64_t seed, int layer, const int32_t* owner,
                            int num_pages, int hkv, int head_dim, int max_pages,
                            const int32_t* ctx_lens, const int32_t* positions,
                            uint64_t heavy_threshold, int heavy_last, const float* unit_dir,
                            cudaStream_t stream) {
  SynthParams p;
  p.cache = static_cast<uint16_t*>(cache);
  p.owner = owner;
  p.ctx_lens = ctx_lens;
  p.positions = positions;
  p.unit_dir = unit_dir;
  p.key_val = stream_key(seed, uint64_t(which == 0 ? 1 : 2) + 16ull * uint64_t(layer));
  p.key_heavy = stream_key(seed, 5ull + 16ull * uint64_t(layer));
  p.heavy_threshold = heavy_threshold;
  p.heavy_last = heavy_last;
  p.is_k = which == 0;
  p.num_pages = num_pages;
  p.hkv = hkv;
  p.head_dim = head_dim;
  p.max_pages = max_pages;
  const size_t chunks = size_t(num_pages) * hkv * 16 * (head_dim / 8);
  const int threads = 256;
  const size_t want = (chunks + threads - 1) / threads;
  const int blocks = int(want < 65536 ? (want ? want : 1) : 65536);
  synth_kv_kernel<<<blocks, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace vegas
