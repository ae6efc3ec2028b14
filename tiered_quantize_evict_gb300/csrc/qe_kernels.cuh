// qe_kernels.cuh -- launch parameters and launchers shared by the host code and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "qe_common.cuh"

namespace qe {

// qe_decode_attn: one layer, all units; see qe_attn.cu
struct AttnParams {
  State st;
  int layer;
  int L;                 // tokens per sequence (after this step's append)
  int nbw;               // bf16 window entries per unit (sink included)
  int nq;                // 2-bit windows per unit
  int cb, cq;            // cost of one 16-token bf16 tile and of one 2-bit window
  long long Cu;          // cost of one unit
  long long C;           // cost of the layer
  int NW;                // warps in the grid
  int pslots;            // partial slots per unit (>= warps whose range meets one unit)
  int ntiles;            // tiles per unit = nbw * w/16 + nq
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
  int L;
  int nbw, nq, ntiles;
  int cb, cq;
  long long Cu, C;
  int NW, pslots;
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
  int L;
  int n_windows;     // windows reached
  int routed_old;    // windows [0, routed_old) entered the pool at earlier events
  int aged_upto;     // windows [0, aged_upto) are complete and older than the recent region
  int kf, kq;
  int exp_nfull, exp_nquant;   // host mirror of the per-unit counts after this event
  Move* moves;
  int* n_moves;
  int max_moves;
};

cudaError_t launch_decode_attn(const AttnParams& p, int grid, cudaStream_t stream);
cudaError_t launch_attn_combine(const CombineParams& p, cudaStream_t stream);
int attn_warps_per_cta();
cudaError_t launch_open_windows(const State& st, int layer, int w_old, int w_new, int nbw_old, cudaStream_t s);
cudaError_t launch_append(const State& st, int layer, int pos0, int n, const uint16_t* k, const uint16_t* v,
                          int n_sm, cudaStream_t s);
cudaError_t launch_route(const RouteParams& p, cudaStream_t s);
cudaError_t launch_moves(const State& st, const Move* moves, const int* n_moves, int n_sm, cudaStream_t s);

}  // namespace qe
