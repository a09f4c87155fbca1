/*
 * kvc_synth.h — seeded synthetic inputs drawn on the device (tests and benchmarks).
 *
 * Not part of the attention path: it fills buffers with the same counter-based draws that the
 * Python module `kvc_synth` makes on the host, so a large workload can be generated in HBM and any
 * element of it redrawn on the host. The generator is Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011); each value is the Irwin-Hall sum of
 * twelve 24-bit uniforms, centred and scaled by 2^-24, rounded once to float32.
 */
#ifndef KVC_SYNTH_H
#define KVC_SYNTH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kvc_synth_fill_normal_f32 — out_dev[i] = std * x(offset + i) for i < n, where x(j) is the draw
 * of element j of stream `stream_id` under key `seed` (counter (j mod 2^32, j >> 32, stream_id, k),
 * k = 0, 1, 2). std == 1 stores x exactly; otherwise the product is rounded to float32 once.
 * Returns 0, or -1 (null pointer) / -4 (CUDA launch error). Asynchronous on `stream`.
 */
int kvc_synth_fill_normal_f32(float* out_dev, size_t n, uint64_t offset, uint64_t seed,
                              uint32_t stream_id, float std, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVC_SYNTH_H */
