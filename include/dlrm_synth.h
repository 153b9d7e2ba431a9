/*
 * dlrm_synth.h -- device-side synthesis of seeded embedding tables.
 *
 * Not part of the method: a helper that fills multi-gigabyte tables on the
 * GPU so that benchmarks and tests need not copy them from the host.  It
 * implements the splitmix64 generator (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) from its published
 * definition; the Python input module implements the same generator
 * independently, and tests check the two bit for bit.
 */
#ifndef DLRM_GB300_SYNTH_H
#define DLRM_GB300_SYNTH_H

#include "dlrm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Element i of d_dst (i in [0, count)) receives the value for global element
 * e = first_elem + i:
 *   z = splitmix64 output number e of the stream seeded with `seed`
 *       (z = mix(seed + (e + 1) * 0x9E3779B97F4A7C15)),
 *   x = (z >> 40) - 2^23                  (signed 24-bit integer, exact in fp32)
 *   v = fp32(x) * fp32(amplitude / 2^23)  (one fp32 rounding)
 * stored as v, or as fp16 of v (round to nearest even); v lies in
 * [-amplitude, amplitude).  For a joint table [rows][D], e = row * D + col.
 *
 *   d_dst  device buffer of `count` elements of dtype (no alignment needed)
 * Returns DLRM_ERR_INVALID_ARG for a null pointer or count < 0.
 */
dlrm_status dlrm_synth_fill_uniform(void* d_dst, dlrm_dtype dtype, uint64_t seed,
                                    int64_t first_elem, int64_t count, double amplitude,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DLRM_GB300_SYNTH_H */
