/*
 * vegas_synth.h - device-side seeded input generator for the Vegas workloads.
 *
 * Not part of the method: it fills a paged K or V cache with the same values
 * the host generator (workload/gen.py) produces for every logical position, so
 * that multi-gigabyte workloads are drawn in HBM in milliseconds.  Definition
 * (identical on both sides, bit for bit):
 *   draw(key, i) = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)   (SplitMix64)
 *   key(seed, tag) = mix64(seed + tag * 0x9E3779B97F4A7C15)
 *   z = float32(u0 + u1 + u2 + u3 - 131070) * float32(sqrt(3)/65536)
 *       with u0..u3 the four 16-bit fields of one draw (Irwin-Hall(4))
 *   K/V element (b, g, pos, j): counter ((b*Hkv + g) << 24 | pos) * d + j,
 *       tag 1 (K) or 2 (V) plus 16 * layer
 *   heavy (K only, pos < L_b): draw(key(seed, 5 + 16*layer), (b*Hkv+g) << 24 | pos)
 *       < heavy_threshold, or pos >= L_b - heavy_last; value 3*u_j + 0.3*z (fp32, RN)
 *   then fp32 -> bf16 round-to-nearest-even.
 */
#ifndef VEGAS_SYNTH_H_
#define VEGAS_SYNTH_H_

#include <stdint.h>
#include "vegas.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Fills cache (device bf16 [num_pages][num_kv_heads][16][head_dim]).
 *   which: 0 = K, 1 = V
 *   owner: device int32 [num_pages]; b * max_pages_per_seq + logical page, or -1
 *          for an unused page (filled with zeros)
 *   ctx_lens: device int32 [batch], L_b
 *   positions: device int32 [batch], positions materialised per sequence;
 *          slots at or past it are zero
 *   unit_dir: device float32 [head_dim], the planted direction u
 */
vegas_status_t vegas_synth_paged_kv(
    void* cache, int which, uint64_t seed, int layer, const int32_t* owner,
    int num_pages, int num_kv_heads, int head_dim, int max_pages_per_seq,
    const int32_t* ctx_lens, const int32_t* positions, uint64_t heavy_threshold,
    int heavy_last, const float* unit_dir, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VEGAS_SYNTH_H_ */
