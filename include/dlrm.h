/*
 * dlrm.h -- C ABI of the GB300 (sm_103a) DLRM embedding + dot-interaction
 * hot path: embedding lookup with sum pooling, dot interaction, interaction
 * backward, and the sparse embedding gradient fused with the SGD row update.
 *
 * The model is the one of the page "DLRM For PyTorch", §Model architecture:
 * one embedding table per categorical feature; the bottom-MLP output and the
 * embedding vectors enter the "dot interaction", whose output is concatenated
 * with the bottom-MLP output and fed to the top MLP.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Names: F = number of tables (categorical features), D = embedding dim
 *    (= bottom-MLP output width), B = batch, nnz = total number of indices,
 *    W = D + F(F+1)/2 = meaningful interaction columns, s = element size.
 *  - Pointers named d_* are DEVICE pointers; h_* are host pointers.  The
 *    caller allocates and owns every buffer; the library allocates nothing,
 *    neither device nor pinned memory.  Scratch space is caller-provided.
 *  - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream).  DLRM_OK means the work was enqueued; there is no
 *    implicit synchronisation and no host<->device copy.
 *  - Errors detectable on the host (null pointers, bad sizes, misalignment,
 *    workspace too small) are returned BEFORE anything is enqueued; nothing is
 *    written.  The message is in dlrm_last_error() (thread-local).
 *  - Errors found on the device are reported as bits OR-ed into *d_status
 *    (a device uint32, may be NULL), read by the caller after synchronising.
 *    No kernel traps; no kernel reads or writes out of bounds.
 *  - Inputs must not alias outputs.  Results are bitwise reproducible for
 *    identical inputs and arguments.
 *  - Tables are one joint row-major buffer [total_rows][D] (the joint layout of
 *    --embedding_type joint*); table t owns rows [row_base[t], row_base[t+1]).
 *  - Index lists are CSR and feature-major: bag (t, b) = indices
 *    [offsets[t*B + b], offsets[t*B + b + 1]).  offsets has F*B + 1 entries,
 *    offsets[0] = 0, non-decreasing, offsets[F*B] = nnz (int32).  This is the
 *    caller's contract (checking it on the host would need a device round
 *    trip); kernels clamp every bag into [0, nnz] and flag
 *    DLRM_STATUS_BAD_OFFSETS, so malformed offsets never cause an access
 *    outside the buffers.
 */
#ifndef DLRM_GB300_H
#define DLRM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DLRM_OK = 0,
    DLRM_ERR_INVALID_ARG = 1,   /* null pointer, negative size, out_cols < W, ... */
    DLRM_ERR_UNSUPPORTED = 2,   /* a legal request this library does not implement */
    DLRM_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (message says which) */
    DLRM_ERR_WORKSPACE = 4,     /* workspace smaller than the size query returned */
    DLRM_ERR_NO_FIT = 5         /* table placement: a table does not fit on its GPU */
} dlrm_status;

typedef enum { DLRM_F32 = 0, DLRM_F16 = 1 } dlrm_dtype;

/* flags */
#define DLRM_FLAG_HASH_INDICES 1u  /* fold every index into its table: idx := ((idx % N_t) + N_t) % N_t
                                      ("DLRM For PyTorch", §Command-line options, --hash_indices) */
#define DLRM_FLAG_POOLED_F16 2u    /* dlrm_emb_fwd: fp32 tables, fp16 pooled output (each bag summed
                                      in fp32, rounded once): the fp16 interaction input of mixed
                                      precision ("DLRM For PyTorch", §Mixed precision training) */
#define DLRM_FLAG_GRAD_F16 4u      /* dlrm_emb_bwd_sgd: grad_pooled is fp16 (from
                                      dlrm_interact_bwd_f16); with a static loss scale S pass lr / S
                                      (exact in fp32 for a power-of-two S such as the pages' 1024) */

/* The most indices (nnz) any entry point takes, 2^31 - 65: index positions, and the kernels'
   32-bit position counters that step up to 32 past them, stay below 2^31.  Larger nnz is
   DLRM_ERR_INVALID_ARG. */
#define DLRM_MAX_NNZ 2147483583LL

/* bits OR-ed into *d_status by kernels */
#define DLRM_STATUS_OOB_INDEX 1u   /* an index outside [0, N_t) with hashing off: it was skipped */
#define DLRM_STATUS_TIMEOUT   2u   /* a bounded on-chip wait gave up; the output is incomplete */
#define DLRM_STATUS_BAD_OFFSETS 4u /* an offset outside [0, nnz] or decreasing: the bag was clamped
                                      into [0, nnz] (results for malformed CSR are unspecified,
                                      but no access leaves the buffers) */

/*
 * dlrm_emb_fwd -- embedding lookup with sum pooling.
 * ("DLRM For PyTorch", §Model architecture: one table per categorical feature
 *  turns each value into a dense vector; §Command-line options:
 *  --embedding_type joint*, --embedding_dim, --hash_indices.)
 *
 *   pooled[b][t][:] = sum_{p in bag(t,b)} tables[row_base[t] + idx'(p)][:]
 *
 * with idx'(p) = indices[p] folded by DLRM_FLAG_HASH_INDICES, or, with hashing
 * off, entries outside [0, N_t) skipped and DLRM_STATUS_OOB_INDEX set.  An
 * empty bag pools to zero.  Sums are accumulated in fp32 in bag order and
 * rounded once to `dtype`; a single-index bag is an exact copy of the row.
 *
 *   d_tables   [total_rows][D] of dtype, 16-byte aligned
 *   d_row_base int64 [F+1], row_base[0] = 0, non-decreasing
 *   d_indices  int32 [nnz];  d_offsets int32 [F*B+1]
 *   d_pooled   [B][F][D] of dtype, 16-byte aligned (output); fp16 with
 *              DLRM_FLAG_POOLED_F16 (fp32 tables only)
 * Requires F >= 1, D >= 1, B >= 0, 0 <= nnz <= DLRM_MAX_NNZ, D*s % 16 == 0.
 */
dlrm_status dlrm_emb_fwd(const void* d_tables, dlrm_dtype dtype, const int64_t* d_row_base,
                         int F, int D, int B, const int32_t* d_indices,
                         const int32_t* d_offsets, int64_t nnz, void* d_pooled,
                         unsigned flags, uint32_t* d_status, void* stream);

/*
 * dlrm_interact_fwd -- dot interaction.
 * ("DLRM For PyTorch", §Model architecture: the bottom-MLP output and the
 *  embedding vectors enter the dot interaction, whose output is concatenated
 *  with the bottom-MLP output; --interaction_op cuda_dot.)
 *
 * For each sample b, Z = [dense[b]; pooled[b][0]; ...; pooled[b][F-1]]
 * ((F+1) x D) and
 *   out[b] = [ dense[b] (D) | z_i . z_j for i = 1..F, j = 0..i-1 (row-major)
 *              | zeros up to out_cols ]
 * Dot products accumulate in fp32 and are rounded once to `dtype`.  For fp16
 * with D % 64 == 0, D <= 256, F <= 32 and 16-byte-aligned rows the products
 * run on the tcgen05 tensor cores; other shapes use CUDA cores.
 *
 *   d_dense  [B][D] of dtype;  d_pooled [B][F][D] of dtype (both 16-byte aligned)
 *   d_out    [B][out_cols] of dtype (output), out_cols >= W
 *   d_status may be NULL; gets DLRM_STATUS_TIMEOUT if a bounded wait gave up.
 * Requires F >= 1, D >= 1, B >= 0, D*s % 16 == 0.
 */
dlrm_status dlrm_interact_fwd(const void* d_dense, const void* d_pooled, dlrm_dtype dtype,
                              int F, int D, int B, void* d_out, int out_cols,
                              uint32_t* d_status, void* stream);

/*
 * dlrm_interact_fwd_cuda_core -- the same operation as dlrm_interact_fwd, always
 * on the CUDA-core (FFMA) kernel, for any shape dlrm_interact_fwd accepts.  It
 * exists to cross-check and time the tensor-core kernel; d_status is not taken
 * because this kernel has no waits.
 */
dlrm_status dlrm_interact_fwd_cuda_core(const void* d_dense, const void* d_pooled, dlrm_dtype dtype,
                                        int F, int D, int B, void* d_out, int out_cols,
                                        void* stream);

/*
 * dlrm_emb_interact_fwd -- dlrm_emb_fwd followed by dlrm_interact_fwd in one
 * pass, for inference: each bag's table row is gathered straight into the
 * tensor-core tile, so the pooled tensor is never written to HBM.
 * (The same two operations as above: "DLRM For PyTorch", §Model
 * architecture; the interaction output is concatenated with the bottom-MLP
 * output.)
 *
 *   out[b] = dlrm_interact_fwd(dense[b], dlrm_emb_fwd(bags of sample b))
 *
 * Results are bit-identical to the two calls (bags of one index are copied,
 * larger bags are summed in fp32 in bag order and rounded once to the table
 * type).  Arguments as in dlrm_emb_fwd and dlrm_interact_fwd.  Shapes taken:
 *   fp16: F <= 32, D a multiple of 64 up to 256, out_cols a multiple of 8
 *         (tensor-core kernel);
 *   fp32: D = 128, F in {8, 26}, out_cols a multiple of 4 and at most
 *         D + 32 * ceil(F(F+1)/2 / 32) (480 for F = 26) (CUDA-core kernel);
 * with 16-byte aligned tables, dense and out; otherwise DLRM_ERR_UNSUPPORTED
 * (use the two calls).  Status bits as in dlrm_emb_fwd, plus
 * DLRM_STATUS_TIMEOUT.  On 1e6-row tables the fp16 pass beats the two calls
 * at 1 to 4 indices per bag (measured); the fp32 pass up to about three,
 * past which the two calls (which need a pooled buffer) are faster, with the
 * same bits.
 */
dlrm_status dlrm_emb_interact_fwd(const void* d_tables, dlrm_dtype dtype, const int64_t* d_row_base,
                                  int F, int D, int B, const int32_t* d_indices,
                                  const int32_t* d_offsets, int64_t nnz, const void* d_dense,
                                  void* d_out, int out_cols, unsigned flags, uint32_t* d_status,
                                  void* stream);

/*
 * dlrm_emb_interact_fwd_train -- the training forward in one pass:
 * dlrm_emb_fwd and dlrm_interact_fwd, also writing the pooled tensor that
 * dlrm_interact_bwd and dlrm_emb_bwd_sgd take.  (The same two operations:
 * "DLRM For PyTorch", §Model architecture.)
 *
 *   d_pooled[b] = dlrm_emb_fwd(bags of sample b)                (output)
 *   d_out[b]    = dlrm_interact_fwd(dense[b], d_pooled[b])      (output)
 *
 * Both are bit-identical to the two calls; the pooled rows are written once
 * and not read back from memory.  Arguments as in dlrm_emb_fwd and
 * dlrm_interact_fwd.  Requires fp32 tables, D = 128, F in {8, 26}, out_cols a
 * multiple of 4 and at most D + 32 * ceil(F(F+1)/2 / 32) (480 for F = 26),
 * 16-byte aligned tables, dense, pooled and out; otherwise
 * DLRM_ERR_UNSUPPORTED (use the two calls).  Flags: DLRM_FLAG_HASH_INDICES.
 * Status bits as in dlrm_emb_fwd.  When nnz exceeds 3 F B (more than three
 * indices per bag on average) the call itself runs the two operations as two
 * launches, which is faster there and gives the same bits.
 */
dlrm_status dlrm_emb_interact_fwd_train(const void* d_tables, dlrm_dtype dtype, const int64_t* d_row_base,
                                        int F, int D, int B, const int32_t* d_indices,
                                        const int32_t* d_offsets, int64_t nnz, const void* d_dense,
                                        void* d_pooled, void* d_out, int out_cols, unsigned flags,
                                        uint32_t* d_status, void* stream);

/*
 * dlrm_interact_bwd -- gradient of dlrm_interact_fwd.
 * With G = grad_out[b][0..W) (pad columns ignored) and M the symmetric
 * (F+1)x(F+1) matrix M_ij = M_ji = G[D + i(i-1)/2 + j] (i > j), M_ii = 0:
 *   dZ = M Z;  grad_dense[b] = G[0..D) + dZ_0;  grad_pooled[b][t] = dZ_{t+1}
 * All arithmetic in fp32 (fp16 inputs are widened exactly).
 *
 *   d_grad_out    fp32 [B][out_cols];  d_dense, d_pooled as in the forward
 *   d_grad_dense  fp32 [B][D] (output);  d_grad_pooled fp32 [B][F][D] (output)
 * All pointers 16-byte aligned.  Requires out_cols >= W, D*s % 16 == 0.
 */
dlrm_status dlrm_interact_bwd(const float* d_grad_out, const void* d_dense,
                              const void* d_pooled, dlrm_dtype dtype, int F, int D, int B,
                              int out_cols, float* d_grad_dense, float* d_grad_pooled,
                              void* stream);

/*
 * dlrm_emb_interact_bwd -- dlrm_interact_bwd for a training step that keeps no
 * pooled tensor: the rows of Z after the dense row are gathered again from the
 * tables, exactly as dlrm_emb_fwd pools them, inside the backward kernel.
 * (The same two operations: "DLRM For PyTorch", §Model architecture -- the
 *  lookup with sum pooling feeds the dot interaction -- and the gradient of
 *  the interaction as stated for dlrm_interact_bwd.)
 *
 *   pooled[b]      = dlrm_emb_fwd(bags of sample b)    (recomputed, not stored)
 *   grad_dense[b], grad_pooled[b] = dlrm_interact_bwd(grad_out[b], dense[b], pooled[b])
 *
 * Results are bit-identical to dlrm_interact_bwd fed the output of dlrm_emb_fwd
 * on the same tables and bags.  Arguments as in dlrm_emb_fwd (tables, row_base,
 * indices, offsets, nnz, flags, d_status) and dlrm_interact_bwd (grad_out,
 * dense, out_cols, grad_dense, grad_pooled).  Requires fp32 tables, D = 128,
 * F in {8, 26}, out_cols a multiple of 4 up to 1024 and 16-byte aligned tables,
 * grad_out, dense, grad_dense and grad_pooled; otherwise DLRM_ERR_UNSUPPORTED
 * (use dlrm_emb_fwd + dlrm_interact_bwd).  Flags: DLRM_FLAG_HASH_INDICES.
 * Status bits as in dlrm_emb_fwd, plus DLRM_STATUS_TIMEOUT.
 */
dlrm_status dlrm_emb_interact_bwd(const void* d_tables, dlrm_dtype dtype, const int64_t* d_row_base,
                                  int F, int D, int B, const int32_t* d_indices,
                                  const int32_t* d_offsets, int64_t nnz, const float* d_grad_out,
                                  const void* d_dense, int out_cols, float* d_grad_dense,
                                  float* d_grad_pooled, unsigned flags, uint32_t* d_status,
                                  void* stream);

/*
 * dlrm_interact_bwd_f16 -- the same gradient for the mixed-precision step
 * ("DLRM For PyTorch", §Mixed precision training: fp16 tensors, static loss
 * scaling, so G and the results carry the loss scale), on the tcgen05 tensor
 * cores: dZ = M Z as one block-diagonal product per four samples, fp32
 * accumulation, each result rounded once to fp16 (grad_dense = G[0..D) +
 * dZ_0 added in fp32 first).
 *
 *   d_grad_out    fp16 [B][out_cols];  d_dense fp16 [B][D];  d_pooled fp16 [B][F][D]
 *   d_grad_dense  fp16 [B][D] (output);  d_grad_pooled fp16 [B][F][D] (output)
 * All pointers 16-byte aligned.  Requires out_cols >= W, a multiple of 8 and
 * at most 1024, F <= 31, D a multiple of 64 up to 256 (DLRM_ERR_UNSUPPORTED
 * otherwise).
 * A device-side wait that times out sets DLRM_STATUS_TIMEOUT in *d_status.
 */
dlrm_status dlrm_interact_bwd_f16(const void* d_grad_out, const void* d_dense, const void* d_pooled, int F,
                                  int D, int B, int out_cols, void* d_grad_dense, void* d_grad_pooled,
                                  uint32_t* d_status, void* stream);

/*
 * Workspace bytes dlrm_emb_bwd_sgd needs for nnz indices of width D over
 * total_rows rows.  Returns 0 for invalid sizes.
 */
size_t dlrm_emb_bwd_sgd_workspace_size(int64_t nnz, int D, int64_t total_rows);

/*
 * dlrm_emb_bwd_sgd -- sparse embedding gradient fused with the SGD update.
 * (The gradient of the sum pooling of dlrm_emb_fwd flows unchanged to every
 *  row of a bag; the tables are FP32 as in "DLRM For PyTorch", §Training
 *  process; the sparse-gradient joint table is --embedding_type joint_sparse.)
 *
 * For every global row r touched by the batch:
 *   g_r = sum over positions p with row(p) = r of grad_pooled[b(p)][t(p)][:]
 *   tables[r] := fmaf(-lr, g_r, tables[r])
 * Rows not touched are left bit-for-bit unchanged; no dense gradient table is
 * formed.  Deterministic: pairs (row, b*F + t) are stably radix-sorted by
 * row; the sorted pairs are cut into items of 256 positions (32 when nnz is
 * at most 8,192), each row's gradients are summed in ascending position order
 * within an item, and the sums of a row that spans several items are
 * combined in item order (a row spanning more than 8 items: 16 contiguous
 * slices of its items, each in order, then the slices in order).  Skipped
 * indices (see dlrm_emb_fwd) contribute nothing.
 *
 *   d_tables       fp32 [total_rows][D], updated in place, 16-byte aligned
 *   d_row_base     int64 [F+1] with row_base[F] = total_rows
 *   total_rows     rows in the joint table, 1 <= total_rows < 2^32 - 1
 *   d_grad_pooled  fp32 [B][F][D] (from dlrm_interact_bwd), 16-byte aligned;
 *                  fp16 with DLRM_FLAG_GRAD_F16 (from dlrm_interact_bwd_f16)
 *   d_workspace    >= dlrm_emb_bwd_sgd_workspace_size(nnz, D, total_rows)
 *                  bytes, 256-byte aligned.  After the stream completes, its
 *                  first nnz uint32 are the sorted row keys (0xFFFFFFFF for
 *                  skipped indices, which sort last) and the nnz uint32 that
 *                  start at byte offset dlrm_ws_align(4*nnz) are the matching
 *                  grad_pooled row numbers b*F + t.
 * Requires D % 4 == 0, at most 1024 (a multiple of 8 with DLRM_FLAG_GRAD_F16).
 */
dlrm_status dlrm_emb_bwd_sgd(float* d_tables, const int64_t* d_row_base, int64_t total_rows,
                             int F, int D, int B, const int32_t* d_indices,
                             const int32_t* d_offsets, int64_t nnz,
                             const void* d_grad_pooled, float lr, void* d_workspace,
                             size_t workspace_bytes, unsigned flags, uint32_t* d_status,
                             void* stream);

/*
 * dlrm_emb_bwd_sgd_noalloc -- dlrm_emb_bwd_sgd for callers that cannot
 * allocate device memory.  (The paper has no counterpart: this is an
 * interface convenience, not part of the method.)
 *
 * Some callers may not call cudaMalloc at all -- for example a plugin run
 * from a host framework's execute callback, where the framework owns every
 * byte of device memory and forbids allocation while it runs -- and cannot
 * hand dlrm_emb_bwd_sgd a workspace either.  This entry point takes the same
 * arguments minus the workspace and uses a scratch array of
 * DLRM_NOALLOC_SCRATCH_BYTES built into the library (a file-scope __device__
 * array; every GPU that loads the library holds it until the process exits).
 * It allocates nothing and calls no allocating routine.
 *
 *  - Sizes whose dlrm_emb_bwd_sgd_workspace_size(nnz, D, total_rows) exceeds
 *    DLRM_NOALLOC_SCRATCH_BYTES are rejected with DLRM_ERR_UNSUPPORTED before
 *    anything is enqueued.  The workspace grows with nnz and D only, so the
 *    limit is at most 809,216 indices at D = 128 and 973,632 at D = 16.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address in the current CUDA context and caches it; make
 *    that first call before any stream capture.  A call from another context
 *    on the device -- for instance after cudaDeviceReset created a new primary
 *    context -- looks the address up again, so it too should come before any
 *    capture.
 *  - All calls share the one array, which keeps the previous call's
 *    contents (everything that must start at zero is cleared by each call).
 *    Calls that overlap on the GPU -- on different streams, or from several
 *    host threads -- race on it and must be serialised by the caller.
 * Results are bit-identical to dlrm_emb_bwd_sgd on the same inputs; the
 * sorted keys are not returned.  Flags as for dlrm_emb_bwd_sgd (with
 * DLRM_FLAG_GRAD_F16 the gradient pointer holds fp16).
 */
#define DLRM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
dlrm_status dlrm_emb_bwd_sgd_noalloc(float* d_tables, const int64_t* d_row_base, int64_t total_rows,
                                     int F, int D, int B, const int32_t* d_indices,
                                     const int32_t* d_offsets, int64_t nnz,
                                     const void* d_grad_pooled, float lr, unsigned flags,
                                     uint32_t* d_status, void* stream);

/*
 * dlrm_set_wait_limit -- how long a bounded on-chip wait of the tensor-core
 * kernels (dlrm_interact_fwd and dlrm_emb_interact_fwd on fp16,
 * dlrm_interact_bwd_f16) lasts before the kernel gives up, in SM clock cycles.
 * (The pages have no counterpart: this is the failure detection of the
 * library itself.)
 *
 * Every wait of those kernels on a copy, a tensor-core product or a peer warp
 * is bounded; when one gives up the kernel lets the copies and products it
 * already issued finish (each within the default bound), frees its tensor
 * memory, sets DLRM_STATUS_TIMEOUT in *d_status and returns, so the context
 * stays usable and the output is incomplete.  The default, about two seconds,
 * only ends a wait that something has broken; a shorter limit exists to test
 * that path (0 gives up at the first wait that is not already complete).
 * cycles < 0 restores the default; larger values are clamped to it.  The limit
 * is read when a call is made (it is a kernel argument) and is process-wide.
 * Returns the previous limit.
 */
int64_t dlrm_set_wait_limit(int64_t cycles);

/* Round a byte count up to the workspace sub-buffer alignment (256 bytes). */
size_t dlrm_ws_align(size_t bytes);

/* Message for the last non-OK return on this thread ("" if none). */
const char* dlrm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DLRM_GB300_H */
