/*
 * flint_synth.h - seeded synthetic inputs on the device.
 *
 * Not part of the method: this draws the random weights and activations that
 * tests and benchmarks feed to the decode layer, so that full-size layers can
 * be made on the GPU while any expert can still be regenerated on the CPU from
 * the same definition.
 *
 * Definition (SplitMix64 of Steele, Lea and Flood, OOPSLA 2014):
 *   mix(z): z = (z ^ z>>30) * 0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB;
 *           return z ^ z>>31                                   (mod 2^64)
 *   u(key, i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)
 *   normal n: twelve 16-bit fields f_j of u(key,3n), u(key,3n+1), u(key,3n+2)
 *   (least significant first); z = (sum_j (2 f_j + 1) - 12*65536) * 2^-17,
 *   exact in float32 (Irwin-Hall sum of twelve uniforms minus 6).
 *   value = float32(z) * sigma (one float32 multiply, nearest even);
 *   bf16 output rounds that value to bf16, nearest even.
 *   stream_key(seed, layer, tensor, expert)
 *     = mix(seed ^ mix(layer<<48 | tensor<<32 | expert)).
 */
#ifndef FLINT_SYNTH_H_
#define FLINT_SYNTH_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 64-bit stream key (host function, no CUDA call). */
uint64_t flint_synth_stream_key(uint64_t seed, uint32_t layer, uint32_t tensor, uint32_t expert);

/* Writes normals start .. start+n-1 of stream `key`, times sigma, to out
 * (device): float32 if out_bf16 == 0, else bf16 bit patterns. Returns 0 on
 * success, 1 on a bad argument, 3 on a CUDA launch error. Asynchronous. */
int flint_synth_normal(uint64_t key, uint64_t start, size_t n, float sigma, int32_t out_bf16,
                       void* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_SYNTH_H_ */
