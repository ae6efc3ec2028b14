// qe_tok_kernels.h -- launchers of the five-tier per-token kernels (qe_tok.cu).
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "qe_tok.cuh"

namespace qe {

cudaError_t tk_prepare(int D);
int tk_attn_warps();
size_t tk_rerank_smem(int D);
// single-token append into the tail (length committed by the next decode step's merge)
cudaError_t tk_launch_append1(const TokState& s, int layer, const uint16_t* k, const uint16_t* v, cudaStream_t st);
// multi-token append (prefill when the layer is empty) with its header update
cudaError_t tk_launch_append(const TokState& s, int layer, int n, bool prefill, const uint16_t* k, const uint16_t* v,
                             int n_sm, cudaStream_t st);
cudaError_t tk_launch_commit_pending(const TokState& s, int layer, int pend, cudaStream_t st);
// attention of one decode step, then its merge (a programmatic dependent of the attention)
// knew / vnew: this step's appended token ([units][head_dim] each, device-accessible), written
// into the tail by the launch itself; null when it is written already
cudaError_t tk_launch_attn(const TokState& s, int layer, int pend, const uint16_t* knew, const uint16_t* vnew,
                           const uint16_t* q, float scale_log2, float* part_o, float2* part_ml, float* logits, int lg_cap,
                           int grid, cudaStream_t st, int debug_expire = 0);
cudaError_t tk_launch_merge(const TokState& s, int layer, int pend, const float* part_o, const float2* part_ml,
                            const float* logits, int lg_cap, int grid, void* out, int out_fp32, cudaStream_t st);
// re-rank of one layer and its header switch
// re-ranks layers [layer0, layer0 + n_layers) in one launch per kernel (scratch slot = layer - layer0)
cudaError_t tk_launch_rerank(const TokState& s, int layer0, int n_layers, cudaStream_t st);

}  // namespace qe
