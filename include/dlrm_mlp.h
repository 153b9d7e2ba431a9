/*
 * dlrm_mlp.h -- the bottom MLP on the tensor cores.
 *
 * "DLRM For PyTorch", §Model architecture: the dense features go through the
 * "bottom MLP", a chain of linear layers with ReLU activations, whose output
 * joins the embedding vectors in the dot interaction; --bottom_mlp_sizes
 * gives 512,256,128 after the 13 numerical features.  Under the pages' mixed
 * precision (§Mixed precision training) the tensors are fp16 with fp32
 * accumulation; here the biases stay fp32 as well.
 *
 * Layer l computes  h_{l+1} = relu(h_l W_l^T + b_l)  (the last layer too),
 * h_0 = x rounded to fp16.  The result is the fp16 `dense` operand of
 * dlrm_interact_fwd / dlrm_emb_interact_fwd.
 *
 * Ownership: every pointer is caller-owned device memory, the call only
 * enqueues work on `stream`.  Errors: DLRM_ERR_INVALID_ARG (sizes, null
 * pointers), DLRM_ERR_UNSUPPORTED (a width that is not a multiple of 16,
 * misaligned pointers), DLRM_ERR_WORKSPACE (ws_bytes below the size query),
 * DLRM_ERR_CUDA.  A device-side wait that times out sets
 * DLRM_STATUS_TIMEOUT in *d_status (when given).
 */
#ifndef DLRM_GB300_MLP_H
#define DLRM_GB300_MLP_H

#include "dlrm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of device workspace dlrm_bottom_mlp_fwd needs for a batch of B and
 * the host array dims[0..n_layers] (0 for invalid arguments): the fp16 copy
 * of x padded to a multiple of 8 columns plus every hidden activation.  The
 * pages' shape (dims[0] <= 16, then 512, 256, 128) runs as one fused launch
 * that reads x directly and keeps the hidden activations on chip: there the
 * workspace is not touched (the size query still counts it). */
size_t dlrm_bottom_mlp_workspace_size(int B, int n_layers, const int* dims);

/* x: fp32 [B][dims[0]].  d_weights: fp16, the layers one after another,
 * layer l as [dims[l+1]][round_up(dims[l], 8)] row-major (PyTorch's Linear
 * layout) with the pad columns zero.  d_biases: fp32, the layers' [dims[l+1]]
 * one after another.  out: fp16 [B][dims[n_layers]].  dims[1..n_layers] must
 * be multiples of 16; all device pointers 16-byte aligned, the workspace
 * 256-byte aligned.  dims is a host array of n_layers + 1 ints. */
dlrm_status dlrm_bottom_mlp_fwd(const float* d_x, int B, int n_layers, const int* dims, const void* d_weights,
                                const float* d_biases, void* d_out, void* d_workspace, size_t ws_bytes,
                                uint32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif
