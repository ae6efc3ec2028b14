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
  const uint16_t* knew;  // pend = 1: the token's K and V [B][Hkv][D] bf16, written by this launch
  const uint16_t* vnew;
  int cb, cq;            // cost of one 16-token bf16 tile and of one 2-bit window
  int pslots;            // partial slots per unit (>= warps whose range meets one unit)
  const uint16_t* q;     // [B][Hq][D] bf16
  float scale_log2;      // log2(e) / sqrt(d)
  float* part_o;         // [units][pslots][G][D] unnormalised output
  float2* part_ml;       // [units][pslots][G] (reference max, sum) in the log2 domain
  float* lse;            // [units][ntiles][G] per-tile log2-sum-exp
  // keys stored pre-RoPE (null: no rotation): cos / sin of 16 b theta_i per 16-token block b
  // [blocks][D/2], and of r theta_i per row offset r < 16 [16][D/2]
  const float2* rope_blk;
  const float2* rope_off;
  // fault injection for tests (qe_debug_inject): k >= 1 makes every warp report its k-th tile
  // wait as expired once that tile's copy has landed; 0: off
  int debug_expire;
};

// qe_attn_combine
struct CombineParams {
  State st;
  int layer;
  int pend;              // as in the attention launch; the combine commits the length
  int cb, cq;
  int NW, pslots;        // warps of the attention launch, partial slots per unit
  const float* part_o;
  const float2* part_ml;
  const float* lse;
  void* out;             // [B][Hq][D] float32 or bf16
  int out_fp32;
  float* delta;          // null: window masses are added to the scores; else written to
                         // delta[unit][window] (a speculative query, committed later or dropped)
};

constexpr int COMBINE_MAXP = 256;   // partials one unit may receive

// One window move decided by a routing event.  A window's exact bf16 copy goes to its host
// store entry the first time the window is kept (Full or Quantized) after leaving the Pinned
// state: a complete window never changes, so a Full window's copy, written when it became Full,
// already serves its first demotion, which then only has to write the ledger.
enum : int {
  MOVE_PACK_COPY = 0,   // Pinned -> Quantized: pack, ledger and exact copy to the host
  MOVE_REUSE = 1,       // -> Quantized again: ledger -> 2-bit slot
  MOVE_PROMOTE = 2,     // Quantized -> Full: exact copy -> bf16 slot
  MOVE_PACK = 3,        // Full -> Quantized, first time: pack and ledger (the exact copy exists)
  MOVE_COPY = 4         // Pinned -> Full: exact copy to the host
};
struct Move {
  int kind;
  int gu;
  int win;
  int src;     // pack / copy: bf16 slot; reuse / promotion: store entry
  int dst;     // pack / reuse: 2-bit slot; promotion: bf16 slot; copy: store entry
  int sent;    // pack: store entry (the exact copy for MOVE_PACK_COPY)
  int wb;      // pack / reuse: store entry whose ledger receives the 2-bit slot's previous codes
               // before the slot is overwritten, or -1
};
// bits of a window's store entry number: its 2-bit codes exist (packed once, held by a 2-bit
// slot or by the host ledger), and the host ledger entry holds them
constexpr int SENT_PACKED = 1 << 29;
constexpr int SENT_LEDGER = 1 << 30;
constexpr int SENT_FLAGS = SENT_PACKED | SENT_LEDGER;

#if defined(__CUDACC__)
// Open window j of unit gu when its first token arrives: take the next free bf16 slot, Pinned,
// score 0, entry nb of the bf16 list.  Returns the slot (-1 and the error flag if the pool is
// empty).
__device__ __forceinline__ int open_window(const State& st, long long gu, int j, int nb) {
  const int head = st.bfree_head[gu];
  if (head >= st.bfree_top[gu] || nb >= st.capb) {
    atomicOr(st.err, ERR_FREELIST);
    return -1;
  }
  const int s = st.bfree[gu * st.capb + head];
  st.bfree_head[gu] = head + 1;
  st.bvictim[gu * st.capb + s] = j;
  st.bslot[gu * st.maxw + j] = s;
  st.tier[gu * st.maxw + j] = TIER_PINNED;
  st.score[gu * st.maxw + j] = 0.f;
  st.blist[gu * st.capb + nb] = make_int2(j, s);
  return s;
}
#endif

// per-unit record of a routing event (same layout as qe_route_diag)
struct RouteDiag {
  int kf, kq, full_old, full_new, full_both, kept_old, kept_new, kept_both, promotions, demotions, evictions;
  float full_cut_kept, full_cut_next, kept_cut_kept, kept_cut_next;
};

struct RouteParams {
  State st;
  int layer;
  Move* moves;
  int* n_moves;
  int max_moves;
  RouteDiag* diag;   // [layers][units]
};

// Fused speculative verify (qe_verify.cu): every draft query of a unit against one read of its
// windows, on the tensor cores.  Rows r = j G + h < 64; the drafts are already appended.
struct VerifyParams {
  State st;
  int layer;
  int L0;                 // length before the drafts (draft j sees positions < L0 + j + 1)
  int n_q;                // drafts
  int R;                  // rows, n_q G <= 64
  int splits;             // CTAs per unit, each over a share of its windows
  const uint16_t* q;      // [n_q][B][Hq][D] bf16
  float scale_log2;       // log2(e) / sqrt(d)
  float* part_o;          // [units][splits][64][D] unnormalised output of each split
  float2* part_ml;        // [units][splits][64] (reference max, sum) in the log2 domain
  float* lse;             // [units][ent_cap][64] per-window log2-sum-exp of each row
  int ent_cap;            // windows (bf16 entries + 2-bit entries) a unit can list
};
cudaError_t launch_verify_attn(const VerifyParams& p, cudaStream_t s);
cudaError_t launch_verify_combine(const VerifyParams& p, void* out, int out_fp32, float* delta, long long qstride,
                                  cudaStream_t s);
cudaError_t prepare_verify_kernels(int D, int W);
int verify_max_rows();
int verify_min_drafts();   // automatic path choice: fused from this many drafts
int verify_max_splits();
int verify_ctas_per_sm(int D, int W);   // resident verify CTAs per SM (tensor memory, shared memory)

cudaError_t launch_decode_attn(const AttnParams& p, int grid, cudaStream_t stream);
int attn_grid(int n_sm, int units, int pslots);
cudaError_t prepare_attn_kernels(int D, int W);
cudaError_t prepare_route_kernels(const State& st);
cudaError_t launch_attn_combine(const CombineParams& p, cudaStream_t stream);
int attn_warps_per_cta();
// mean CUDA-event time (us) of n empty launches shaped like the attention launch (synchronous)
cudaError_t time_empty_attn_launch(int D, int W, int grid, int n, cudaStream_t stream, double* us);
cudaError_t launch_verify_commit(const State& st, int layer, int L0, int n_q, int n_accept, const float* delta,
                                 long long qstride, cudaStream_t s);
// tok_major: k and v are [n][units][D] (token-major, as a verify's drafts) instead of [units][n][D]
cudaError_t launch_append(const State& st, int layer, int n, const uint16_t* k, const uint16_t* v, int n_sm,
                          cudaStream_t s, bool tok_major = false);
// routes layers [p.layer, p.layer + n_layers) in one launch
cudaError_t launch_route(const RouteParams& p, int n_layers, cudaStream_t s);
cudaError_t launch_commit_length(const State& st, int layer, int n, cudaStream_t s);
cudaError_t launch_moves(const State& st, const Move* moves, const int* n_moves, int n_sm, cudaStream_t s);

}  // namespace qe
