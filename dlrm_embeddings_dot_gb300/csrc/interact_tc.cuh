// interact_tc.cuh -- tensor-core (tcgen05) dot interaction for fp16 inputs.
#pragma once

#include "common.cuh"

namespace dlrm {

// True when the fp16 interaction of this shape can run on the tcgen05 kernel:
// 1 <= F <= 32, D a multiple of 64 up to 256, 16-byte output rows up to 2048
// columns, all base pointers 16-byte aligned.
bool tc_interact_supported(int F, int D, int out_cols, const void* dense, const void* pooled,
                           const void* out);

dlrm_status tc_interact_fwd(const void* dense, const void* pooled, int F, int D, int B, void* out,
                            int out_cols, uint32_t* status, cudaStream_t stream);

}  // namespace dlrm
