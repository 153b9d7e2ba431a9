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
 *   u = ((z >> 40) + 0.5) / 2^24                      (double, exact)
 *   v = u * (hi - lo), then v + lo                    (two rounded double ops, no FMA)
 *   stored as (float)v, or as fp16 of (float)v (round to nearest even).
 * For a joint table [rows][D], element e = row * D + col.
 *
 *   d_dst  device buffer of `count` elements of dtype (no alignment needed)
 * Returns DLRM_ERR_INVALID_ARG for a null pointer or count < 0.
 */
dlrm_status dlrm_synth_fill_uniform(void* d_dst, dlrm_dtype dtype, uint64_t seed,
                                    int64_t first_elem, int64_t count, double lo, double hi,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DLRM_GB300_SYNTH_H */
