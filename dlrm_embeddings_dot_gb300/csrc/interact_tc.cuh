// interact_tc.cuh -- internal entry points shared by the interaction sources:
// the tensor-core (tcgen05) interaction for fp16 inputs and the fp32
// register-kernel lookup + interaction.
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

// True when the fp32 lookup + interaction can run in one pass on the register
// kernel: D = 128, F in {8, 26}, out_cols a multiple of 4 and at most
// D + 32 * ceil(F(F+1)/2 / 32), 16-byte-aligned tables, dense, pooled
// (or null) and out.
bool regs_emb_interact_supported(int F, int D, int out_cols, const void* tables, const void* dense,
                                 const void* pooled, const void* out);

// The fp32 lookup + interaction in one pass; pooled (may be null) receives
// the pooled rows, bit-identical to the lookup's.
dlrm_status regs_emb_interact_fwd(const float* tables, const int64_t* row_base, int F, int D, int B,
                                  const int32_t* indices, const int32_t* offsets, int64_t nnz, const float* dense,
                                  float* pooled, float* out, int out_cols, bool hash, uint32_t* status,
                                  cudaStream_t stream);

}  // namespace dlrm
