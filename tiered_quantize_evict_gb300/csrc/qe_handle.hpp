// qe_handle.hpp -- the handle behind the C ABI (internal; shared by the library's host files).
#pragma once
#include <string>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "qe.h"
#include "qe_kernels.cuh"
#include "qe_tok.cuh"

namespace qe {

// An NVTX range over one call of the ABI (header-only NVTX v3: without a profiler attached,
// a push or pop is one test of a null function pointer).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Host shadow of a layer's device header (launch shapes never depend on it; checks and
// introspection do).
struct LayerMirror {
  int L = 0;
  int pending = 0;    // single-token appends whose length the device has not committed yet
  const uint16_t* pk = nullptr;   // pending token's K and V (device): written by the next decode step
  const uint16_t* pv = nullptr;
  int routed_upto = 0;
  int n_full = 0;
  int n_quant = 0;
  int kf = 0, kq = 0;
  int verify_n = 0;    // > 0: a speculative verify of that many drafts awaits qe_verify_commit
  int verify_L0 = 0;   // length before the drafts
};

// Host shadow of a five-tier layer.
struct TokMirror {
  int L = 0;
  int n_tail = 0;     // tail tokens, the pending one included
  int pending = 0;    // appended token whose length the next decode step's merge commits
  // the pending token's K and V (device-accessible) while it is not written yet: the next
  // decode step's attention writes it, any other call first writes it with its own launch
  const uint16_t* pk = nullptr;
  const uint16_t* pv = nullptr;
};

}  // namespace qe

struct qe_handle_s {
  qe_config cfg{};
  cudaStream_t stream = nullptr;
  int device = 0;
  int n_sm = 0;
  qe::State st{};
  std::vector<qe::LayerMirror> lay;
  int units = 0;
  long long gu_total = 0;
  // scratch for the attention split-K
  float* part_o = nullptr;
  float2* part_ml = nullptr;
  float* lse = nullptr;
  int pslots_cap = 0;         // partial slots per unit
  int attn_grid = 0;          // CTAs of every attention launch (fixed)
  int ntiles_cap = 0;
  // moves
  qe::Move* moves = nullptr;
  int* n_moves = nullptr;
  int max_moves = 0;
  qe::RouteDiag* diag = nullptr;   // [n_layers][units] latest routing event of each layer
  // staging for host pointers
  uint16_t* tok_stage = nullptr;   // [n_layers][2][units][D]: single-token appends from host memory
  void* stage[4] = {nullptr, nullptr, nullptr, nullptr};
  size_t stage_bytes[4] = {0, 0, 0, 0};
  // pinned host store
  void* hstore_host = nullptr;
  void* hledger_host = nullptr;
  // speculative verify: window masses of each draft query, [n_layers][verify_cap][units][maxw]
  float* vdelta = nullptr;
  int verify_cap = 0;
  // fused verify scratch (grown on first use, outside any capture): per-split partials and
  // per-window log2-sum-exps of the up to 64 draft x head rows
  float* vf_part_o = nullptr;
  float2* vf_part_ml = nullptr;
  float* vf_lse = nullptr;
  int vf_splits = 0;
  // keys stored pre-RoPE: angle tables (null when rope_theta == 0)
  float2* rope_blk = nullptr;   // [ceil(max_context / 16)][D/2] cos, sin of 16 b theta_i
  float2* rope_off = nullptr;   // [16][D/2] cos, sin of r theta_i
  // tile costs of the split-K partition
  int cost_b = 8, cost_q = 6;
  // timing
  bool timing = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  double timed_bytes = 0;
  long long timed_launches = 0;
  long long launches = 0;
  int debug_expire = 0;   // qe_debug_inject(QE_DEBUG_EXPIRE_WAIT): applies to the next decode step
  int verify_path = 0;    // qe_debug_inject(QE_DEBUG_VERIFY_PATH): 0 automatic, 1 fused, 2 per draft
  std::string err;
  // five-tier per-token mode (cfg.tiering == QE_TIERING_TOKENS)
  bool tok = false;
  qe::TokState ts{};
  std::vector<qe::TokMirror> tlay;
  float* tk_part_o = nullptr;
  float2* tk_part_ml = nullptr;
  float* tk_logits = nullptr;
  int tk_grid = 0;
  int tk_lgcap = 0;
  std::vector<void*> tk_allocs;   // every device allocation of the mode
};

namespace qe {
// qe_debug_inject(QE_DEBUG_FAIL_DEVICE_ALLOC): true when this device allocation of qe_init is
// the one chosen to fail (qe_host.cu); qe_init restarts the count
bool inject_alloc_failure();
void inject_begin_init();
const char* injected_note();   // " (injected by qe_debug_inject)" once after an injected failure, else ""
// five-tier mode (qe_tok_host.cu)
qe_status tok_init(const qe_config& c, cudaStream_t stream, qe_handle* out, std::string& err);
void tok_free(qe_handle h);
qe_status tok_append(qe_handle h, int layer, const void* k, const void* v, int n, int flags);
qe_status tok_decode(qe_handle h, int layer, const void* q, void* out, int flags);
qe_status tok_route(qe_handle h, int layer);
qe_status tok_layer_info(qe_handle h, int layer, qe_layer_info* info);
}  // namespace qe
