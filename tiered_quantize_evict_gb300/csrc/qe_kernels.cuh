// qe_kernels.cuh -- launch parameters and launchers shared by the host code and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "qe_common.cuh"

namespace qe {

// qe_decode_attn: one layer, all units; see qe_attn.cu.  Step-dependent counts come from the
// device-resident layer header; every field here is fixed for the handle's lifetime except
// the buffers, which the caller may keep fixed too.
struct AttnParams {
  State st;
  int layer;
  int pend;              // single-token appends not yet counted in the header's length (0 or 1)
  int* lay_out;          // [4]: length, bf16 entries, 2-bit entries, tiles per unit, for the combine
  int cb, cq;            // cost of one 16-token bf16 tile and of one 2-bit window
  int pslots;            // partial slots per unit (>= warps whose range meets one unit)
  const uint16_t* q;     // [B][Hq][D] bf16
  float scale_log2;      // log2(e) / sqrt(d)
  float* part_o;         // [units][pslots][G][D] unnormalised output
  float2* part_ml;       // [units][pslots][G] (reference max, sum) in the log2 domain
  float* lse;            // [units][ntiles][G] per-tile log2-sum-exp
};

// qe_attn_combine
struct CombineParams {
  State st;
  int layer;
  const int* lay_in;     // written by the attention launch; the combine commits the length
  int cb, cq;
  int NW, pslots;        // warps of the attention launch, partial slots per unit
  const float* part_o;
  const float2* part_ml;
  const float* lse;
  void* out;             // [B][Hq][D] float32 or bf16
  int out_fp32;
};

constexpr int COMBINE_MAXP = 256;   // partials one unit may receive

// one window move decided by a routing event
struct Move {
  int kind;    // 0 pack (first demotion), 1 ledger reuse, 2 promotion
  int gu;
  int win;
  int src;     // pack: bf16 slot; reuse/promotion: store entry
  int dst;     // pack/reuse: 2-bit slot; promotion: bf16 slot
  int sent;    // pack: store entry to fill
};

struct RouteParams {
  State st;
  int layer;
  Move* moves;
  int* n_moves;
  int max_moves;
};

cudaError_t launch_decode_attn(const AttnParams& p, int grid, cudaStream_t stream);
int attn_grid(int n_sm, int units, int pslots);
cudaError_t prepare_attn_kernels(int D, int W);
cudaError_t prepare_route_kernels(const State& st);
cudaError_t launch_attn_combine(const CombineParams& p, cudaStream_t stream);
int attn_warps_per_cta();
cudaError_t launch_append(const State& st, int layer, int n, const uint16_t* k, const uint16_t* v, int n_sm,
                          cudaStream_t s);
cudaError_t launch_route(const RouteParams& p, cudaStream_t s);
cudaError_t launch_commit_length(const State& st, int layer, int n, cudaStream_t s);
cudaError_t launch_moves(const State& st, const Move* moves, const int* n_moves, int n_sm, cudaStream_t s);

}  // namespace qe
