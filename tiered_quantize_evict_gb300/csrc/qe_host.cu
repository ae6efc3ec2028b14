// qe_host.cu -- C ABI (include/qe.h): handle, device pools, host mirror, launches.
//
// The host keeps a mirror of the per-layer counts that every unit shares (all sequences of a
// layer have the same length, so after each routing event every unit has the same number of
// Full, Quantized and Pinned windows); launch shapes are computed from it without reading the
// device.  Window identities, slots, scores and codes live only on the device.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qe.h"
#include "qe_handle.hpp"
#include "qe_kernels.cuh"

namespace {

using qe::LayerMirror;

thread_local std::string g_init_error;

// qe_debug_inject: the device allocation of the next qe_init that fails (1-based, 0 none), the
// count of device allocations the current qe_init has made, and whether the next pinned host
// store allocation fails.  Process-wide and one-shot.
std::atomic<int> g_fail_alloc_nth{0};
std::atomic<int> g_alloc_count{0};
std::atomic<int> g_fail_host_store{0};
std::atomic<int> g_fired{0};   // an injected allocation failure has fired and is not yet reported

}  // namespace

namespace qe {
void inject_begin_init() { g_alloc_count.store(0); }
bool inject_alloc_failure() {
  const int n = g_fail_alloc_nth.load();
  if (n <= 0) return false;
  if (g_alloc_count.fetch_add(1) + 1 != n) return false;
  g_fail_alloc_nth.store(0);
  g_fired.store(1);
  return true;
}
const char* injected_note() { return g_fired.exchange(0) ? " (injected by qe_debug_inject)" : ""; }
}  // namespace qe

namespace {

qe_status fail(qe_handle h, qe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->err = buf; else g_init_error = buf;
  return s;
}

#define QE_CK(h, call)                                                                            \
  do {                                                                                            \
    cudaError_t e_ = (call);                                                                      \
    if (e_ != cudaSuccess)                                                                        \
      return fail((h), e_ == cudaErrorMemoryAllocation ? QE_ERR_OOM : QE_ERR_CUDA, "%s: %s (%s:%d)", #call, \
                  cudaGetErrorString(e_), __FILE__, __LINE__);                                    \
  } while (0)

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

int qslot_bytes(int w, int d) { return 2 * (w * d / 4) + 8 * d + 8 * w; }

// Capacity rule, see qe.h (qe::capacities_at: double precision, no fused operations)
void capacities(const qe_config& c, int L, int& kf, int& kq) {
  qe::CapCfg cc{c.cap_mode, c.kf, c.kq, c.frac_bf16, c.frac_int2, c.budget_frac};
  qe::capacities_at(cc, c.n_sink, c.n_recent, c.window, c.head_dim, L, kf, kq);
}

template <class T>
qe_status dalloc(qe_handle h, T** p, size_t count, const char* what) {
  if (qe::inject_alloc_failure())
    return fail(h, QE_ERR_OOM, "cudaMalloc of %s (%zu bytes) failed%s", what, count * sizeof(T), qe::injected_note());
  cudaError_t e = cudaMalloc((void**)p, count * sizeof(T) > 0 ? count * sizeof(T) : 16);
  if (e != cudaSuccess)
    return fail(h, QE_ERR_OOM, "cudaMalloc of %s (%zu bytes) failed: %s", what, count * sizeof(T), cudaGetErrorString(e));
  return QE_OK;
}

qe_status check_layer(qe_handle h, int layer) {
  if (!h) return QE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->cfg.n_layers) return fail(h, QE_ERR_INVALID_ARG, "layer %d out of range", layer);
  return QE_OK;
}

qe_status ensure_stage(qe_handle h, int i, size_t bytes) {
  if (h->stage_bytes[i] >= bytes) return QE_OK;
  if (h->stage[i]) cudaFree(h->stage[i]);
  h->stage[i] = nullptr;
  h->stage_bytes[i] = 0;
  QE_CK(h, cudaMalloc(&h->stage[i], bytes));
  h->stage_bytes[i] = bytes;
  return QE_OK;
}

void fill_info(qe_handle h, const LayerMirror& m, qe_layer_info* info);

// The device address of a page-locked, device-mapped host buffer, aligned to `align` bytes;
// nullptr for pageable memory (which goes through copies).  Kernels read and write such a buffer
// over the host link in stream order, exactly where a copy would have run.
const void* mapped_view(const void* p, size_t align) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  if (reinterpret_cast<uintptr_t>(a.devicePointer) % align) return nullptr;
  return a.devicePointer;
}

// a single-token append that no decode step consumed: write the token and advance the device
// length now
qe_status commit_pending(qe_handle h, int layer) {
  LayerMirror& m = h->lay[layer];
  if (!m.pending) return QE_OK;
  QE_CK(h, qe::launch_append(h->st, layer, 1, m.pk, m.pv, h->n_sm, h->stream));
  QE_CK(h, qe::launch_commit_length(h->st, layer, m.pending, h->stream));
  h->launches += 2;
  m.pending = 0;
  m.pk = m.pv = nullptr;
  return QE_OK;
}

int nbw_of(const qe_handle h, const LayerMirror& m) {
  const int nwin = ceil_div(m.L, h->cfg.window);
  return 1 + m.n_full + (nwin - m.routed_upto);
}

void free_all(qe_handle h) {
  qe::State& s = h->st;
  void* ptrs[] = {s.tier, s.bslot, s.qslot, s.sent, s.score, s.blist, s.qlist, s.bfree, s.bfree_head, s.bfree_top,
                  s.qfree, s.qfree_top, s.sfree, s.sfree_top, s.bvictim, s.qvictim, s.bprev, s.qprev, s.bslab, s.qslab, s.qrange, s.err, s.stats, s.ldev, h->part_o, h->part_ml,
                  h->lse, h->moves, h->n_moves, h->stage[0], h->stage[1], h->stage[2], h->stage[3],
                  h->tok_stage, h->diag, h->rope_blk, h->rope_off, h->vdelta, h->vf_part_o, h->vf_part_ml,
                  h->vf_lse};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (h->hstore_host) cudaFreeHost(h->hstore_host);
  if (h->hledger_host) cudaFreeHost(h->hledger_host);
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
}

}  // namespace

extern "C" {

const char* qe_last_error(qe_handle h) { return h ? h->err.c_str() : g_init_error.c_str(); }

long long qe_kernel_launches(qe_handle h) { return h ? h->launches : 0; }

qe_status qe_init(const qe_config* cfg, void* cuda_stream, qe_handle* out) {
  qe::NvtxRange nvtx_("qe_init");
  if (!cfg || !out) return fail(nullptr, QE_ERR_INVALID_ARG, "null argument");
  qe::inject_begin_init();
  const qe_config& c = *cfg;
  if (c.batch < 1 || c.n_layers < 1 || c.n_kv_heads < 1 || c.n_q_heads < 1 || c.n_q_heads % c.n_kv_heads)
    return fail(nullptr, QE_ERR_INVALID_ARG, "bad head/batch/layer counts");
  const int G = c.n_q_heads / c.n_kv_heads;
  if (G != 1 && G != 2 && G != 4) return fail(nullptr, QE_ERR_INVALID_ARG, "query heads per KV head must be 1, 2 or 4");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(nullptr, QE_ERR_INVALID_ARG, "head_dim must be 64 or 128");
  if (c.tiering != QE_TIERING_WINDOWS && c.tiering != QE_TIERING_TOKENS)
    return fail(nullptr, QE_ERR_INVALID_ARG, "tiering must be QE_TIERING_WINDOWS or QE_TIERING_TOKENS");
  if (c.max_context < 1) return fail(nullptr, QE_ERR_INVALID_ARG, "bad max_context");
  if (!(c.rope_theta >= 0.0)) return fail(nullptr, QE_ERR_INVALID_ARG, "rope_theta must be >= 0");
  if (c.tiering == QE_TIERING_TOKENS && c.rope_theta != 0.0)
    return fail(nullptr, QE_ERR_INVALID_ARG, "pre-RoPE keys are served by the window tiering only");
  if (c.tiering == QE_TIERING_TOKENS) {
    std::string err;
    qe_status ts = qe::tok_init(c, static_cast<cudaStream_t>(cuda_stream), out, err);
    if (ts != QE_OK) g_init_error = err;
    return ts;
  }
  if (c.window != 16 && c.window != 32 && c.window != 64) return fail(nullptr, QE_ERR_INVALID_ARG, "window must be 16, 32 or 64");
  if (c.n_sink < 0 || c.n_sink >= c.window || c.n_sink >= 16) return fail(nullptr, QE_ERR_INVALID_ARG, "need 0 <= n_sink < min(window, 16)");
  if (c.n_recent < 1) return fail(nullptr, QE_ERR_INVALID_ARG, "n_recent must be >= 1");
  if (c.max_context < 1 || c.cap_mode < 0 || c.cap_mode > 2) return fail(nullptr, QE_ERR_INVALID_ARG, "bad max_context or cap_mode");
  if (c.cap_mode == 0 && (c.kf < 0 || c.kq < 0)) return fail(nullptr, QE_ERR_INVALID_ARG, "kf, kq must be >= 0");
  if (c.int2_slack < -1) return fail(nullptr, QE_ERR_INVALID_ARG, "int2_slack must be >= -1");

  qe_handle h = new qe_handle_s();
  h->cfg = c;
  h->stream = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    delete h;
    return fail(nullptr, QE_ERR_CUDA, "no CUDA device: %s", cudaGetErrorString(e));
  }
  h->cost_q = h->cost_q * c.window / 32 > 0 ? h->cost_q * c.window / 32 : 1;

  const int maxw = ceil_div(c.max_context, c.window);
  if (maxw > 4096) {
    delete h;
    return fail(nullptr, QE_ERR_INVALID_ARG, "max_context / window must be <= 4096 windows");
  }
  int kf_max = 0, kq_max = 0;
  capacities(c, c.max_context, kf_max, kq_max);
  h->units = c.batch * c.n_kv_heads;
  h->gu_total = (long long)h->units * c.n_layers;
  qe::State& st = h->st;
  st.units = h->units;
  st.n_layers = c.n_layers;
  st.maxw = maxw;
  st.capb = 1 + maxw;
  // the 2-bit slab holds K_q windows plus slack: a freed slot keeps its window's codes until it
  // is handed out again (oldest first), so a window that returns soon takes its codes back and
  // a kept window's ledger reaches the host only when its codes are about to be overwritten
  {
    const int slack = c.int2_slack == 0 ? (kq_max / 2 > 16 ? kq_max / 2 : 16) : (c.int2_slack < 0 ? 0 : c.int2_slack);
    st.capq = kq_max > 0 ? kq_max + slack : 1;
  }
  st.caps = (kf_max + kq_max) > 0 ? kf_max + kq_max : 1;
  if (st.caps > maxw) st.caps = maxw;
  if (st.capq > maxw) st.capq = maxw;
  st.n_sink = c.n_sink;
  st.n_recent = c.n_recent;
  st.G = G;
  st.Hq = c.n_q_heads;
  st.Hkv = c.n_kv_heads;
  st.geo.D = c.head_dim;
  st.geo.W = c.window;
  st.cap = qe::CapCfg{c.cap_mode, c.kf, c.kq, c.frac_bf16, c.frac_int2, c.budget_frac};
  st.max_context = c.max_context;
  h->lay.assign(c.n_layers, LayerMirror{});

  const long long GU = h->gu_total;
  const size_t bslot_b = (size_t)st.geo.bslot_bytes(), qslot_b = (size_t)st.geo.qslot_bytes();
  qe_status s;
#define QE_ALLOC(ptr, n, what)                              \
  if ((s = dalloc(h, &(ptr), (size_t)(n), what)) != QE_OK) { \
    std::string m = h->err;                                 \
    free_all(h);                                            \
    delete h;                                               \
    g_init_error = m;                                       \
    return s;                                               \
  }
  QE_ALLOC(st.tier, GU * maxw, "tier");
  QE_ALLOC(st.bslot, GU * maxw, "bslot");
  QE_ALLOC(st.qslot, GU * maxw, "qslot");
  QE_ALLOC(st.sent, GU * maxw, "sent");
  QE_ALLOC(st.score, GU * maxw, "score");
  QE_ALLOC(st.blist, GU * st.capb, "blist");
  QE_ALLOC(st.qlist, GU * st.capq, "qlist");
  QE_ALLOC(st.bfree, GU * st.capb, "bfree");
  QE_ALLOC(st.bfree_head, GU, "bfree_head");
  QE_ALLOC(st.bfree_top, GU, "bfree_top");
  QE_ALLOC(st.bvictim, GU * st.capb, "bvictim");
  QE_ALLOC(st.qvictim, GU * st.capq, "qvictim");
  QE_ALLOC(st.bprev, GU * maxw, "bprev");
  QE_ALLOC(st.qprev, GU * maxw, "qprev");
  QE_ALLOC(st.qfree, GU * st.capq, "qfree");
  QE_ALLOC(st.qfree_top, GU, "qfree_top");
  QE_ALLOC(st.sfree, GU * st.caps, "sfree");
  QE_ALLOC(st.sfree_top, GU, "sfree_top");
  QE_ALLOC(st.bslab, GU * st.capb * bslot_b, "bf16 window pool");
  QE_ALLOC(st.qslab, GU * st.capq * qslot_b, "2-bit window pool");
  QE_ALLOC(st.qrange, GU * st.capq, "2-bit slot ranges");
  QE_ALLOC(st.err, 1, "error flag");
  QE_ALLOC(st.stats, (size_t)c.n_layers * qe::N_STATS, "stats");
  QE_ALLOC(st.ldev, (size_t)c.n_layers, "layer headers");

  // split-K scratch: one CTA per SM, attn_warps_per_cta() warps each; a unit meets at most
  // NW / units + 2 warp ranges
  const int NW = h->n_sm * qe::attn_warps_per_cta();
  h->pslots_cap = NW / h->units + 3;
  if (h->pslots_cap > qe::COMBINE_MAXP) h->pslots_cap = qe::COMBINE_MAXP;
  h->attn_grid = qe::attn_grid(h->n_sm, h->units, h->pslots_cap);
  h->ntiles_cap = st.capb * (c.window / 16) + st.capq;
  QE_ALLOC(h->part_o, (size_t)h->units * h->pslots_cap * G * c.head_dim, "partials");
  QE_ALLOC(h->part_ml, (size_t)h->units * h->pslots_cap * G, "partial stats");
  QE_ALLOC(h->lse, (size_t)h->units * h->ntiles_cap * G, "tile log-sum-exp");
  QE_ALLOC(h->diag, (size_t)c.n_layers * h->units, "routing records");
  QE_ALLOC(h->tok_stage, (size_t)c.n_layers * 2 * h->units * c.head_dim, "token staging");
  {
    const long long mm = (long long)c.n_layers * h->units * st.caps + 16;   // one event of every layer
    if (mm > 0x7FFFFFFFLL) {
      free_all(h);
      delete h;
      return fail(nullptr, QE_ERR_OOM, "move list of %lld entries exceeds the int range", mm);
    }
    h->max_moves = (int)mm;
  }
  {
    void* mp = nullptr;
    if (qe::inject_alloc_failure() || cudaMalloc(&mp, (size_t)h->max_moves * sizeof(qe::Move)) != cudaSuccess) {
      free_all(h);
      delete h;
      return fail(nullptr, QE_ERR_OOM, "cudaMalloc of the move list failed%s", qe::injected_note());
    }
    h->moves = static_cast<qe::Move*>(mp);
  }
  QE_ALLOC(h->n_moves, 1, "move count");
#undef QE_ALLOC

  // pinned host backing store, mapped into the device address space
  const bool inj_store = g_fail_host_store.exchange(0) != 0;
  e = inj_store ? cudaErrorMemoryAllocation
                : cudaHostAlloc(&h->hstore_host, (size_t)GU * st.caps * bslot_b, cudaHostAllocMapped);
  if (e == cudaSuccess) e = cudaHostAlloc(&h->hledger_host, (size_t)GU * st.caps * qslot_b, cudaHostAllocMapped);
  void* dstore = nullptr;
  void* dledger = nullptr;
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(&dstore, h->hstore_host, 0);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(&dledger, h->hledger_host, 0);
  if (e != cudaSuccess) {
    std::string m = std::string("pinned host store: ") + cudaGetErrorString(e) + (inj_store ? " (injected by qe_debug_inject)" : "");
    free_all(h);
    delete h;
    g_init_error = m;
    return QE_ERR_HOST_STORE;
  }
  st.hstore = static_cast<uint8_t*>(dstore);
  st.hledger = static_cast<uint8_t*>(dledger);

  // initial table: nothing reached; free stacks hold every slot (bf16 slot 0 is the sink's)
  cudaError_t ie = cudaSuccess;
  auto set = [&](cudaError_t x) { if (ie == cudaSuccess) ie = x; };
  set(cudaMemsetAsync(st.tier, 0, GU * maxw, h->stream));
  set(cudaMemsetAsync(st.bslot, 0xFF, GU * maxw * 4, h->stream));
  set(cudaMemsetAsync(st.qslot, 0xFF, GU * maxw * 4, h->stream));
  set(cudaMemsetAsync(st.sent, 0xFF, GU * maxw * 4, h->stream));
  set(cudaMemsetAsync(st.score, 0, GU * maxw * 4, h->stream));
  set(cudaMemsetAsync(st.bslab, 0, GU * st.capb * bslot_b, h->stream));
  set(cudaMemsetAsync(st.qslab, 0, GU * st.capq * qslot_b, h->stream));
  set(cudaMemsetAsync(st.qrange, 0, GU * st.capq * 4, h->stream));
  set(cudaMemsetAsync(st.err, 0, 4, h->stream));
  set(cudaMemsetAsync(h->diag, 0, (size_t)c.n_layers * h->units * sizeof(qe::RouteDiag), h->stream));
  set(cudaMemsetAsync(st.stats, 0, (size_t)c.n_layers * qe::N_STATS * 8, h->stream));
  set(cudaMemsetAsync(st.bvictim, 0xFF, GU * st.capb * 4, h->stream));
  set(cudaMemsetAsync(st.qvictim, 0xFF, GU * st.capq * 4, h->stream));
  set(cudaMemsetAsync(st.bprev, 0xFF, GU * maxw * 4, h->stream));
  set(cudaMemsetAsync(st.qprev, 0xFF, GU * maxw * 4, h->stream));
  set(cudaMemsetAsync(st.bfree_head, 0, GU * 4, h->stream));
  set(cudaMemsetAsync(st.ldev, 0, (size_t)c.n_layers * sizeof(qe::LayerDev), h->stream));
  {
    std::vector<int> tmp;
    tmp.resize((size_t)GU * st.capb);
    for (long long gu = 0; gu < GU; ++gu)
      for (int i = 0; i < st.capb - 1; ++i) tmp[gu * st.capb + i] = 1 + i;   // slot 0 is the sink's
    set(cudaMemcpy(st.bfree, tmp.data(), tmp.size() * 4, cudaMemcpyHostToDevice));
    std::vector<int> top(GU, st.capb - 1);
    set(cudaMemcpy(st.bfree_top, top.data(), GU * 4, cudaMemcpyHostToDevice));
    tmp.assign((size_t)GU * st.capq, 0);
    for (long long gu = 0; gu < GU; ++gu)
      for (int i = 0; i < st.capq; ++i) tmp[gu * st.capq + i] = i;
    set(cudaMemcpy(st.qfree, tmp.data(), tmp.size() * 4, cudaMemcpyHostToDevice));
    top.assign(GU, st.capq);
    set(cudaMemcpy(st.qfree_top, top.data(), GU * 4, cudaMemcpyHostToDevice));
    tmp.assign((size_t)GU * st.caps, 0);
    for (long long gu = 0; gu < GU; ++gu)
      for (int i = 0; i < st.caps; ++i) tmp[gu * st.caps + i] = st.caps - 1 - i;
    set(cudaMemcpy(st.sfree, tmp.data(), tmp.size() * 4, cudaMemcpyHostToDevice));
    top.assign(GU, st.caps);
    set(cudaMemcpy(st.sfree_top, top.data(), GU * 4, cudaMemcpyHostToDevice));
    std::vector<int2> bl((size_t)GU * st.capb, make_int2(-1, -1));
    for (long long gu = 0; gu < GU; ++gu) bl[gu * st.capb] = make_int2(-1, 0);
    set(cudaMemcpy(st.blist, bl.data(), bl.size() * sizeof(int2), cudaMemcpyHostToDevice));
  }
  if (c.rope_theta > 0.0) {
    // angle tables in double precision, rounded once: theta_i = base^(-2i/d); block b holds
    // the angle 16 b theta_i, offset r the angle r theta_i
    // every 16-token block of every window slot (a tile is only read where it holds a valid row)
    const int half = c.head_dim / 2, nblk = ceil_div(c.max_context, c.window) * (c.window / 16) + 1;
    std::vector<float2> blk((size_t)nblk * half), off(16 * (size_t)half);
    for (int i = 0; i < half; ++i) {
      const double th = std::pow(c.rope_theta, -2.0 * i / c.head_dim);
      for (int b = 0; b < nblk; ++b) {
        const double a = 16.0 * b * th;
        blk[(size_t)b * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
      for (int r = 0; r < 16; ++r) off[(size_t)r * half + i] = make_float2((float)std::cos(r * th), (float)std::sin(r * th));
    }
    void* pb = nullptr;
    void* po = nullptr;
    set(qe::inject_alloc_failure() ? cudaErrorMemoryAllocation : cudaMalloc(&pb, blk.size() * sizeof(float2)));
    set(qe::inject_alloc_failure() ? cudaErrorMemoryAllocation : cudaMalloc(&po, off.size() * sizeof(float2)));
    h->rope_blk = static_cast<float2*>(pb);
    h->rope_off = static_cast<float2*>(po);
    if (ie == cudaSuccess) set(cudaMemcpy(pb, blk.data(), blk.size() * sizeof(float2), cudaMemcpyHostToDevice));
    if (ie == cudaSuccess) set(cudaMemcpy(po, off.data(), off.size() * sizeof(float2), cudaMemcpyHostToDevice));
  }
  set(qe::prepare_attn_kernels(c.head_dim, c.window));
  set(qe::prepare_verify_kernels(c.head_dim, c.window));
  set(qe::prepare_route_kernels(st));
  set(cudaStreamSynchronize(h->stream));
  if (ie != cudaSuccess) {
    std::string m = std::string("initialising the cache: ") + cudaGetErrorString(ie) + qe::injected_note();
    free_all(h);
    delete h;
    g_init_error = m;
    return ie == cudaErrorMemoryAllocation ? QE_ERR_OOM : QE_ERR_CUDA;
  }
  *out = h;
  return QE_OK;
}

qe_status qe_destroy(qe_handle h) {
  if (!h) return QE_ERR_INVALID_ARG;
  cudaStreamSynchronize(h->stream);
  if (h->tok) {
    qe::tok_free(h);
    delete h;
    return QE_OK;
  }
  free_all(h);
  delete h;
  return QE_OK;
}

qe_status qe_append(qe_handle h, int layer, const void* k, const void* v, int n_tokens, int flags) {
  qe::NvtxRange nvtx_("qe_append");
  if (h && h->tok) return qe::tok_append(h, layer, k, v, n_tokens, flags);
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if (h->lay[layer].verify_n) return fail(h, QE_ERR_STATE, "layer %d awaits qe_verify_commit", layer);
  if (!k || !v || n_tokens < 1) return fail(h, QE_ERR_INVALID_ARG, "append needs K, V and n_tokens >= 1");
  LayerMirror& m = h->lay[layer];
  if (m.L + n_tokens > h->cfg.max_context)
    return fail(h, QE_ERR_CAPACITY, "append of %d tokens passes max_context %d (length %d)", n_tokens,
                h->cfg.max_context, m.L);
  if ((s = commit_pending(h, layer)) != QE_OK) return s;
  const size_t bytes = (size_t)h->units * n_tokens * h->cfg.head_dim * 2;
  const uint16_t* kd = static_cast<const uint16_t*>(k);
  const uint16_t* vd = static_cast<const uint16_t*>(v);
  if (n_tokens == 1) {
    // The next decode step of this layer writes the token (inside its attention launch) and its
    // combine commits the length.  That launch reads a pinned host token in place; a pageable
    // one waits in the layer's own staging slots.
    if (flags & QE_HOST_PTRS) {
      const void* mk = mapped_view(k, 4);
      const void* mv = mapped_view(v, 2);
      if (mk && mv) {
        kd = static_cast<const uint16_t*>(mk);
        vd = static_cast<const uint16_t*>(mv);
      } else {
        uint16_t* ks = h->tok_stage + (size_t)layer * 2 * h->units * h->cfg.head_dim;
        uint16_t* vs = ks + (size_t)h->units * h->cfg.head_dim;
        QE_CK(h, cudaMemcpyAsync(ks, k, bytes, cudaMemcpyHostToDevice, h->stream));
        QE_CK(h, cudaMemcpyAsync(vs, v, bytes, cudaMemcpyHostToDevice, h->stream));
        kd = ks;
        vd = vs;
      }
    }
    m.pending = 1;
    m.pk = kd;
    m.pv = vd;
    m.L += 1;
    return QE_OK;
  }
  if (flags & QE_HOST_PTRS) {
    if ((s = ensure_stage(h, 0, bytes)) != QE_OK || (s = ensure_stage(h, 1, bytes)) != QE_OK) return s;
    QE_CK(h, cudaMemcpyAsync(h->stage[0], k, bytes, cudaMemcpyHostToDevice, h->stream));
    QE_CK(h, cudaMemcpyAsync(h->stage[1], v, bytes, cudaMemcpyHostToDevice, h->stream));
    kd = static_cast<const uint16_t*>(h->stage[0]);
    vd = static_cast<const uint16_t*>(h->stage[1]);
  }
  QE_CK(h, qe::launch_append(h->st, layer, n_tokens, kd, vd, h->n_sm, h->stream));
  h->launches += 2;
  m.L += n_tokens;
  return QE_OK;
}

static qe_status decode_impl(qe_handle h, int layer, const void* q, void* out, int flags, float* delta);

qe_status qe_decode_step(qe_handle h, int layer, const void* q, void* out, int flags) {
  qe::NvtxRange nvtx_("qe_decode_step");
  if (h && h->tok) return qe::tok_decode(h, layer, q, out, flags);
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if (h->lay[layer].verify_n) return fail(h, QE_ERR_STATE, "layer %d awaits qe_verify_commit", layer);
  return decode_impl(h, layer, q, out, flags, nullptr);
}

// one decode step; delta non-null: the window masses go to delta (a speculative query)
static qe_status decode_impl(qe_handle h, int layer, const void* q, void* out, int flags, float* delta) {
  qe_status s;
  if (!q || !out) return fail(h, QE_ERR_INVALID_ARG, "decode needs q and out");
  LayerMirror& m = h->lay[layer];
  if (m.L < 1) return fail(h, QE_ERR_STATE, "decode on an empty layer");
  const qe_config& c = h->cfg;
  const int D = c.head_dim;
  const size_t qbytes = (size_t)c.batch * c.n_q_heads * D * 2;
  const size_t obytes = (size_t)c.batch * c.n_q_heads * D * (c.out_fp32 ? 4 : 2);
  const uint16_t* qd = static_cast<const uint16_t*>(q);
  void* od = out;
  bool out_copy = false;   // pageable output: combine into staging, then copy out
  if (flags & QE_HOST_PTRS) {
    if (const void* mq = mapped_view(q, 4)) {
      qd = static_cast<const uint16_t*>(mq);   // the attention warps read a pinned query in place
    } else {
      if ((s = ensure_stage(h, 2, qbytes)) != QE_OK) return s;
      QE_CK(h, cudaMemcpyAsync(h->stage[2], q, qbytes, cudaMemcpyHostToDevice, h->stream));
      qd = static_cast<const uint16_t*>(h->stage[2]);
    }
    if (const void* mo = mapped_view(out, c.out_fp32 ? 4 : 2)) {
      od = const_cast<void*>(mo);   // the combine writes a pinned output in place
    } else {
      if ((s = ensure_stage(h, 3, obytes)) != QE_OK) return s;
      od = h->stage[3];
      out_copy = true;
    }
  }
  qe::AttnParams p{};
  p.st = h->st;
  p.layer = layer;
  p.pend = m.pending;
  p.knew = m.pk;
  p.vnew = m.pv;
  m.pending = 0;
  m.pk = m.pv = nullptr;
  p.cb = h->cost_b;
  p.cq = h->cost_q;
  p.pslots = h->pslots_cap;
  p.q = qd;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  p.part_o = h->part_o;
  p.part_ml = h->part_ml;
  p.lse = h->lse;
  p.rope_blk = h->rope_blk;
  p.rope_off = h->rope_off;
  p.debug_expire = h->debug_expire;
  h->debug_expire = 0;   // one step only
  {
    const int sub = c.window / 16;
    const int ntiles = nbw_of(h, m) * sub + m.n_quant;
    if (ntiles > h->ntiles_cap) return fail(h, QE_ERR_CAPACITY, "tile count %d exceeds %d", ntiles, h->ntiles_cap);
  }
  const int grid = h->attn_grid;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  unsigned ev_flags = cudaEventRecordDefault;
  if (h->timing) {
    while (h->ev_pool.size() < h->ev_used + 2) {
      cudaEvent_t ev;
      QE_CK(h, cudaEventCreate(&ev));
      h->ev_pool.push_back(ev);
    }
    e0 = h->ev_pool[h->ev_used];
    e1 = h->ev_pool[h->ev_used + 1];
    h->ev_used += 2;
    // inside a stream capture the records must be external to happen when the graph runs
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    QE_CK(h, cudaStreamIsCapturing(h->stream, &cs));
    ev_flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    QE_CK(h, cudaEventRecordWithFlags(e0, h->stream, ev_flags));
  }
  QE_CK(h, qe::launch_decode_attn(p, grid, h->stream));
  ++h->launches;
  if (h->timing) {
    QE_CK(h, cudaEventRecordWithFlags(e1, h->stream, ev_flags));
    h->timed_launches += 1;
    qe_layer_info info;
    fill_info(h, m, &info);   // host shadow: no synchronisation inside the timed path
    h->timed_bytes += info.attn_bytes;
  }
  qe::CombineParams cp{};
  cp.st = h->st;
  cp.layer = layer;
  cp.pend = p.pend;
  cp.cb = p.cb;
  cp.cq = p.cq;
  cp.NW = grid * qe::attn_warps_per_cta();
  cp.pslots = p.pslots;
  cp.part_o = h->part_o;
  cp.part_ml = h->part_ml;
  cp.lse = h->lse;
  cp.out = od;
  cp.out_fp32 = c.out_fp32;
  cp.delta = delta;
  QE_CK(h, qe::launch_attn_combine(cp, h->stream));
  ++h->launches;
  if (out_copy) QE_CK(h, cudaMemcpyAsync(out, od, obytes, cudaMemcpyDeviceToHost, h->stream));
  return QE_OK;
}

// qe_verify's fused path: append the drafts in one launch (the length becomes L0 + n_q), then
// one attention launch over (unit, split) and one combine launch writing every draft's output
// and its window masses into dl.
static qe_status verify_fused(qe_handle h, int layer, const void* q, const void* k, const void* v, void* out, int n_q,
                              int flags, float* dl) {
  qe_status s;
  LayerMirror& m = h->lay[layer];
  const qe_config& c = h->cfg;
  const int D = c.head_dim;
  const size_t kv_bytes = (size_t)n_q * h->units * D * 2;
  const size_t q_bytes = (size_t)n_q * c.batch * c.n_q_heads * D * 2;
  const size_t o_bytes = (size_t)n_q * c.batch * c.n_q_heads * D * (c.out_fp32 ? 4 : 2);
  const uint16_t* kd = static_cast<const uint16_t*>(k);
  const uint16_t* vd = static_cast<const uint16_t*>(v);
  const uint16_t* qd = static_cast<const uint16_t*>(q);
  void* od = out;
  if (flags & QE_HOST_PTRS) {   // every buffer through the handle's staging
    if ((s = ensure_stage(h, 0, kv_bytes)) != QE_OK || (s = ensure_stage(h, 1, kv_bytes)) != QE_OK ||
        (s = ensure_stage(h, 2, q_bytes)) != QE_OK || (s = ensure_stage(h, 3, o_bytes)) != QE_OK)
      return s;
    QE_CK(h, cudaMemcpyAsync(h->stage[0], k, kv_bytes, cudaMemcpyHostToDevice, h->stream));
    QE_CK(h, cudaMemcpyAsync(h->stage[1], v, kv_bytes, cudaMemcpyHostToDevice, h->stream));
    QE_CK(h, cudaMemcpyAsync(h->stage[2], q, q_bytes, cudaMemcpyHostToDevice, h->stream));
    kd = static_cast<const uint16_t*>(h->stage[0]);
    vd = static_cast<const uint16_t*>(h->stage[1]);
    qd = static_cast<const uint16_t*>(h->stage[2]);
    od = h->stage[3];
  }
  // splits: the fewest that fill the resident CTA slots in nearly whole waves (a partial last
  // wave leaves SMs idle for a whole CTA's time)
  const int slots = h->n_sm * qe::verify_ctas_per_sm(D, c.window);
  int splits = 1;
  double best = -1.0;
  for (int sp = 1; sp <= qe::verify_max_splits(); ++sp) {
    const long long ctas = (long long)h->units * sp;
    const long long waves = (ctas + slots - 1) / slots;
    const double eff = (double)ctas / (double)(waves * slots);
    if (eff > best + 1e-9) {
      best = eff;
      splits = sp;
    }
    if (ctas >= slots && eff >= 0.9) break;
  }
  const int rows = qe::verify_max_rows();
  const int ent_cap = h->st.capb + h->st.capq;
  if (!h->vf_part_o || h->vf_splits < splits) {
    if (h->vf_part_o) cudaFree(h->vf_part_o);
    if (h->vf_part_ml) cudaFree(h->vf_part_ml);
    if (h->vf_lse) cudaFree(h->vf_lse);
    h->vf_part_o = nullptr;
    h->vf_part_ml = nullptr;
    h->vf_lse = nullptr;
    h->vf_splits = 0;
    if ((s = dalloc(h, &h->vf_part_o, (size_t)h->units * splits * rows * D, "verify partials")) != QE_OK ||
        (s = dalloc(h, &h->vf_part_ml, (size_t)h->units * splits * rows, "verify partial stats")) != QE_OK ||
        (s = dalloc(h, &h->vf_lse, (size_t)h->units * ent_cap * rows, "verify window sums")) != QE_OK)
      return s;
    h->vf_splits = splits;
  }
  QE_CK(h, qe::launch_append(h->st, layer, n_q, kd, vd, h->n_sm, h->stream, true));
  h->launches += 2;
  qe::VerifyParams vp{};
  vp.st = h->st;
  vp.layer = layer;
  vp.L0 = m.L;
  vp.n_q = n_q;
  vp.R = n_q * h->st.G;
  vp.splits = splits;
  vp.q = qd;
  vp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  vp.part_o = h->vf_part_o;
  vp.part_ml = h->vf_part_ml;
  vp.lse = h->vf_lse;
  vp.ent_cap = ent_cap;
  // the attention launch is timed like a decode step's (qe_set_timing)
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  unsigned ev_flags = cudaEventRecordDefault;
  if (h->timing) {
    while (h->ev_pool.size() < h->ev_used + 2) {
      cudaEvent_t ev;
      QE_CK(h, cudaEventCreate(&ev));
      h->ev_pool.push_back(ev);
    }
    e0 = h->ev_pool[h->ev_used];
    e1 = h->ev_pool[h->ev_used + 1];
    h->ev_used += 2;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    QE_CK(h, cudaStreamIsCapturing(h->stream, &cs));
    ev_flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    QE_CK(h, cudaEventRecordWithFlags(e0, h->stream, ev_flags));
  }
  QE_CK(h, qe::launch_verify_attn(vp, h->stream));
  if (h->timing) {
    QE_CK(h, cudaEventRecordWithFlags(e1, h->stream, ev_flags));
    h->timed_launches += 1;
    LayerMirror mm = m;
    mm.L += n_q;   // the drafts are appended
    qe_layer_info info;
    fill_info(h, mm, &info);
    h->timed_bytes += info.attn_bytes;
  }
  QE_CK(h, qe::launch_verify_combine(vp, od, c.out_fp32, dl, (long long)h->units * h->st.maxw, h->stream));
  h->launches += 2;
  if (od != out) QE_CK(h, cudaMemcpyAsync(out, od, o_bytes, cudaMemcpyDeviceToHost, h->stream));
  m.verify_L0 = m.L;
  m.L += n_q;
  m.verify_n = n_q;
  return QE_OK;
}

qe_status qe_verify(qe_handle h, int layer, const void* q, const void* k, const void* v, void* out, int n_q,
                    int flags) {
  qe::NvtxRange nvtx_("qe_verify");
  if (h && h->tok) return fail(h, QE_ERR_STATE, "speculative verify serves window-tiered handles");
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  LayerMirror& m = h->lay[layer];
  if (m.verify_n) return fail(h, QE_ERR_STATE, "layer %d awaits qe_verify_commit", layer);
  if (!q || !k || !v || !out || n_q < 1 || n_q > QE_VERIFY_MAX)
    return fail(h, QE_ERR_INVALID_ARG, "verify needs q, k, v, out and 1 <= n_q <= %d", QE_VERIFY_MAX);
  if (m.L < 1) return fail(h, QE_ERR_STATE, "verify on an empty layer");
  const qe_config& c = h->cfg;
  if (m.L + m.pending + n_q > c.max_context)
    return fail(h, QE_ERR_CAPACITY, "%d drafts pass max_context %d", n_q, c.max_context);
  if ((s = commit_pending(h, layer)) != QE_OK) return s;
  if (n_q > h->verify_cap) {
    // window masses of each draft query; grown outside any stream capture
    if (h->vdelta) cudaFree(h->vdelta);
    h->vdelta = nullptr;
    h->verify_cap = 0;
    QE_CK(h, cudaMalloc(&h->vdelta, (size_t)c.n_layers * n_q * h->units * h->st.maxw * sizeof(float)));
    h->verify_cap = n_q;
  }
  const long long qstride = (long long)h->units * h->st.maxw;
  float* dl = h->vdelta + (size_t)layer * h->verify_cap * qstride;
  QE_CK(h, cudaMemsetAsync(dl, 0, (size_t)n_q * qstride * sizeof(float), h->stream));
  // All drafts against one read of the cache on the tensor cores, when the rows fit one mma tile
  // and the keys are used as stored (keys stored pre-RoPE verify draft by draft).  The fused
  // launch costs about as much as five decode steps whatever the number of rows (32K context,
  // head_dim 128), so by default it serves five drafts or more.
  const int rows = n_q * h->st.G;
  const bool fused_ok = !h->rope_blk && rows <= qe::verify_max_rows();
  const bool fused = fused_ok && (h->verify_path == 1 || (h->verify_path == 0 && n_q >= qe::verify_min_drafts()));
  if (fused) return verify_fused(h, layer, q, k, v, out, n_q, flags, dl);
  const int D = c.head_dim;
  const size_t kv_tok = (size_t)h->units * D * 2;                       // one draft's K (or V)
  const size_t q_tok = (size_t)c.batch * c.n_q_heads * D * 2;           // one draft's queries
  const size_t o_tok = (size_t)c.batch * c.n_q_heads * D * (c.out_fp32 ? 4 : 2);
  m.verify_L0 = m.L;
  for (int j = 0; j < n_q; ++j) {
    const char* kj = static_cast<const char*>(k) + j * kv_tok;
    const char* vj = static_cast<const char*>(v) + j * kv_tok;
    if ((s = qe_append(h, layer, kj, vj, 1, flags)) != QE_OK) return s;
    if ((s = decode_impl(h, layer, static_cast<const char*>(q) + j * q_tok, static_cast<char*>(out) + j * o_tok, flags,
                         dl + j * qstride)) != QE_OK)
      return s;
  }
  m.verify_n = n_q;
  return QE_OK;
}

qe_status qe_verify_commit(qe_handle h, int layer, int n_accept) {
  qe::NvtxRange nvtx_("qe_verify_commit");
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  LayerMirror& m = h->lay[layer];
  if (!m.verify_n) return fail(h, QE_ERR_STATE, "layer %d has no verify to commit", layer);
  if (n_accept < 0 || n_accept > m.verify_n)
    return fail(h, QE_ERR_INVALID_ARG, "n_accept %d outside [0, %d]", n_accept, m.verify_n);
  const long long qstride = (long long)h->units * h->st.maxw;
  QE_CK(h, qe::launch_verify_commit(h->st, layer, m.verify_L0, m.verify_n, n_accept,
                                    h->vdelta + (size_t)layer * h->verify_cap * qstride, qstride, h->stream));
  ++h->launches;
  m.L = m.verify_L0 + n_accept;
  m.verify_n = 0;
  return QE_OK;
}

// Checks one layer before a routing event and returns its new mirror values; launches nothing
// but the commit of a pending append.
static qe_status route_check(qe_handle h, int layer, LayerMirror& next) {
  if (h->lay[layer].verify_n) return fail(h, QE_ERR_STATE, "layer %d awaits qe_verify_commit", layer);
  qe_status s0 = commit_pending(h, layer);
  if (s0 != QE_OK) return s0;
  const LayerMirror& m = h->lay[layer];
  const qe_config& c = h->cfg;
  int aged = (m.L - c.n_recent) >= 0 ? (m.L - c.n_recent) / c.window : 0;
  if (aged < m.routed_upto) aged = m.routed_upto;
  int kf, kq;
  capacities(c, m.L, kf, kq);
  if (kq > h->st.capq) return fail(h, QE_ERR_CAPACITY, "Kq %d exceeds the 2-bit pool (%d)", kq, h->st.capq);
  const int ncand = m.n_full + m.n_quant + (aged - m.routed_upto);
  const int nf = kf < ncand ? kf : ncand;
  const int nq = kq < ncand - nf ? kq : ncand - nf;
  if (nf + nq > h->st.caps) return fail(h, QE_ERR_CAPACITY, "kept windows %d exceed the host store (%d)", nf + nq, h->st.caps);
  next = m;
  next.routed_upto = aged;
  next.n_full = nf;
  next.n_quant = nq;
  next.kf = kf;
  next.kq = kq;
  return QE_OK;
}

// Routes layers [l0, l0 + n): every layer is checked first (nothing is routed if one fails),
// then one route launch covers all of them and one move launch carries out their moves.
static qe_status route_layers(qe_handle h, int l0, int n) {
  std::vector<LayerMirror> next((size_t)n);
  for (int i = 0; i < n; ++i) {
    qe_status s = route_check(h, l0 + i, next[(size_t)i]);
    if (s != QE_OK) return s;
  }
  qe::RouteParams p{};
  p.st = h->st;
  p.layer = l0;
  p.moves = h->moves;
  p.n_moves = h->n_moves;
  p.max_moves = h->max_moves;
  p.diag = h->diag;
  QE_CK(h, cudaMemsetAsync(h->n_moves, 0, 4, h->stream));
  QE_CK(h, qe::launch_route(p, n, h->stream));
  QE_CK(h, qe::launch_moves(h->st, h->moves, h->n_moves, h->n_sm, h->stream));
  h->launches += 2;
  for (int i = 0; i < n; ++i) h->lay[(size_t)(l0 + i)] = next[(size_t)i];
  return QE_OK;
}

qe_status qe_route(qe_handle h, int layer) {
  qe::NvtxRange nvtx_("qe_route");
  if (!h) return QE_ERR_INVALID_ARG;
  if (h->tok) return qe::tok_route(h, layer);
  if (layer == -1) return route_layers(h, 0, h->cfg.n_layers);
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  return route_layers(h, layer, 1);
}

qe_status qe_synchronize(qe_handle h) {
  qe::NvtxRange nvtx_("qe_synchronize");
  if (!h) return QE_ERR_INVALID_ARG;
  QE_CK(h, cudaStreamSynchronize(h->stream));
  unsigned flag = 0;
  QE_CK(h, cudaMemcpy(&flag, h->st.err, 4, cudaMemcpyDeviceToHost));
  if (flag)
    return fail(h, flag & qe::ERR_TIMEOUT ? QE_ERR_TIMEOUT : QE_ERR_DEVICE,
                "device consistency flag 0x%x (1 free list, 2 table, 4 wait timeout, 8 count mismatch, 16 move list)",
                flag);
  return QE_OK;
}

}  // extern "C"

namespace {
void fill_info(qe_handle h, const LayerMirror& m, qe_layer_info* info) {
  const qe_config& c = h->cfg;
  info->length = m.L;
  info->n_windows = ceil_div(m.L, c.window);
  info->routed_upto = m.routed_upto;
  info->n_full = m.n_full;
  info->n_quant = m.n_quant;
  info->n_pinned = info->n_windows - m.routed_upto;
  info->kf = m.kf;
  info->kq = m.kq;
  info->max_windows = h->st.maxw;
  info->units = h->units;
  // bf16 tokens present: sink + Full windows (complete) + Pinned windows (window 0 and the
  // current window partial).  A Full window 0 holds w - n_sink tokens; counting it as w
  // overstates the bytes by at most n_sink tokens per unit.
  double tok = std::min(c.n_sink, m.L);
  tok += (double)m.n_full * c.window;
  for (int j = m.routed_upto; j < info->n_windows; ++j) {
    const int lo = j == 0 ? c.n_sink : 0;
    const int hi = std::min(c.window, m.L - j * c.window);
    if (hi > lo) tok += hi - lo;
  }
  info->attn_bytes = (tok * 4.0 * c.head_dim + (double)m.n_quant * qslot_bytes(c.window, c.head_dim)) * h->units;
}
}  // namespace

extern "C" {

qe_status qe_get_layer_info(qe_handle h, int layer, qe_layer_info* info) {
  if (h && h->tok) {
    if (!info) return fail(h, QE_ERR_INVALID_ARG, "null info");
    return qe::tok_layer_info(h, layer, info);
  }
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if ((s = commit_pending(h, layer)) != QE_OK) return s;
  if (!info) return fail(h, QE_ERR_INVALID_ARG, "null info");
  // the device header is authoritative (it also advances under CUDA-graph replays)
  QE_CK(h, cudaStreamSynchronize(h->stream));
  qe::LayerDev d{};
  QE_CK(h, cudaMemcpy(&d, h->st.ldev + layer, sizeof d, cudaMemcpyDeviceToHost));
  LayerMirror m;
  m.L = d.L;
  m.routed_upto = d.routed_upto;
  m.n_full = d.n_full;
  m.n_quant = d.n_quant;
  m.kf = d.kf;
  m.kq = d.kq;
  m.verify_n = h->lay[layer].verify_n;     // a pending verify stays pending
  m.verify_L0 = h->lay[layer].verify_L0;
  h->lay[layer] = m;   // resynchronise the host shadow
  fill_info(h, m, info);
  return QE_OK;
}

qe_status qe_get_tiers(qe_handle h, int layer, uint8_t* host, size_t bytes) {
  if (h && h->tok) return fail(h, QE_ERR_STATE, "a window-tier call on a token-tiered handle");
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if ((s = commit_pending(h, layer)) != QE_OK) return s;
  const size_t need = (size_t)h->units * h->st.maxw;
  if (!host || bytes < need) return fail(h, QE_ERR_INVALID_ARG, "tier buffer needs %zu bytes", need);
  QE_CK(h, cudaStreamSynchronize(h->stream));
  QE_CK(h, cudaMemcpy(host, h->st.tier + (size_t)layer * need, need, cudaMemcpyDeviceToHost));
  return QE_OK;
}

qe_status qe_get_scores(qe_handle h, int layer, float* host, size_t bytes) {
  if (h && h->tok) return fail(h, QE_ERR_STATE, "a window-tier call on a token-tiered handle");
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if ((s = commit_pending(h, layer)) != QE_OK) return s;
  const size_t n = (size_t)h->units * h->st.maxw;
  if (!host || bytes < n * 4) return fail(h, QE_ERR_INVALID_ARG, "score buffer needs %zu bytes", n * 4);
  QE_CK(h, cudaStreamSynchronize(h->stream));
  QE_CK(h, cudaMemcpy(host, h->st.score + (size_t)layer * n, n * 4, cudaMemcpyDeviceToHost));
  return QE_OK;
}

qe_status qe_set_scores(qe_handle h, int layer, const float* host, size_t bytes) {
  if (h && h->tok) return fail(h, QE_ERR_STATE, "a window-tier call on a token-tiered handle");
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if ((s = commit_pending(h, layer)) != QE_OK) return s;
  const size_t n = (size_t)h->units * h->st.maxw;
  if (!host || bytes < n * 4) return fail(h, QE_ERR_INVALID_ARG, "score buffer needs %zu bytes", n * 4);
  QE_CK(h, cudaStreamSynchronize(h->stream));
  QE_CK(h, cudaMemcpy(h->st.score + (size_t)layer * n, host, n * 4, cudaMemcpyHostToDevice));
  return QE_OK;
}

static qe_status read_int(qe_handle h, const int* dptr, int* out) {
  QE_CK(h, cudaMemcpy(out, dptr, 4, cudaMemcpyDeviceToHost));
  return QE_OK;
}

qe_status qe_get_quant_window(qe_handle h, int layer, int unit, int window, uint8_t* k_codes, uint8_t* v_codes,
                              float* k_min, float* k_scale, float* v_min, float* v_scale) {
  if (h && h->tok) return fail(h, QE_ERR_STATE, "a window-tier call on a token-tiered handle");
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if (unit < 0 || unit >= h->units || window < 0 || window >= h->st.maxw)
    return fail(h, QE_ERR_INVALID_ARG, "unit or window out of range");
  QE_CK(h, cudaStreamSynchronize(h->stream));
  const long long gu = (long long)layer * h->units + unit;
  uint8_t tier = 0;
  QE_CK(h, cudaMemcpy(&tier, h->st.tier + gu * h->st.maxw + window, 1, cudaMemcpyDeviceToHost));
  if (tier != QE_TIER_QUANT) return fail(h, QE_ERR_STATE, "window %d is not Quantized (tier %d)", window, tier);
  int slot = -1;
  if ((s = read_int(h, h->st.qslot + gu * h->st.maxw + window, &slot)) != QE_OK) return s;
  if (slot < 0 || slot >= h->st.capq) return fail(h, QE_ERR_DEVICE, "bad 2-bit slot %d", slot);
  const qe::Geo g = h->st.geo;
  std::vector<uint8_t> buf(g.qslot_bytes());
  QE_CK(h, cudaMemcpy(buf.data(), h->st.qslab + (gu * h->st.capq + slot) * (long long)g.qslot_bytes(), buf.size(),
                      cudaMemcpyDeviceToHost));
  for (int r = 0; r < g.W; ++r)
    for (int c = 0; c < g.D; ++c) {
      qe::CodePos pk = qe::kcode_pos(g, r, c), pv = qe::vcode_pos(g, r, c);
      unsigned wk, wv;
      memcpy(&wk, buf.data() + pk.byte, 4);
      memcpy(&wv, buf.data() + pv.byte, 4);
      if (k_codes) k_codes[r * g.D + c] = (wk >> pk.bit) & 3u;
      if (v_codes) v_codes[r * g.D + c] = (wv >> pv.bit) & 3u;
    }
  for (int c = 0; c < g.D; ++c) {
    if (k_min) memcpy(k_min + c, buf.data() + g.off_kmin() + 4 * qe::kparam_pos(c), 4);
    if (k_scale) memcpy(k_scale + c, buf.data() + g.off_kscale() + 4 * qe::kparam_pos(c), 4);
  }
  for (int r = 0; r < g.W; ++r) {
    if (v_min) memcpy(v_min + r, buf.data() + g.off_vmin() + 4 * qe::vparam_pos(g, r), 4);
    if (v_scale) memcpy(v_scale + r, buf.data() + g.off_vscale() + 4 * qe::vparam_pos(g, r), 4);
  }
  return QE_OK;
}

qe_status qe_get_bf16_window(qe_handle h, int layer, int unit, int window, uint16_t* k, uint16_t* v) {
  if (h && h->tok) return fail(h, QE_ERR_STATE, "a window-tier call on a token-tiered handle");
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if (unit < 0 || unit >= h->units || window < -1 || window >= h->st.maxw)
    return fail(h, QE_ERR_INVALID_ARG, "unit or window out of range");
  QE_CK(h, cudaStreamSynchronize(h->stream));
  const long long gu = (long long)layer * h->units + unit;
  int slot = 0;
  if (window >= 0) {
    uint8_t tier = 0;
    QE_CK(h, cudaMemcpy(&tier, h->st.tier + gu * h->st.maxw + window, 1, cudaMemcpyDeviceToHost));
    if (tier != QE_TIER_PINNED && tier != QE_TIER_FULL)
      return fail(h, QE_ERR_STATE, "window %d is not in bf16 (tier %d)", window, tier);
    if ((s = read_int(h, h->st.bslot + gu * h->st.maxw + window, &slot)) != QE_OK) return s;
  }
  if (slot < 0 || slot >= h->st.capb) return fail(h, QE_ERR_DEVICE, "bad bf16 slot %d", slot);
  const qe::Geo g = h->st.geo;
  std::vector<uint8_t> buf(g.bslot_bytes());
  QE_CK(h, cudaMemcpy(buf.data(), h->st.bslab + (gu * h->st.capb + slot) * (long long)g.bslot_bytes(), buf.size(),
                      cudaMemcpyDeviceToHost));
  for (int r = 0; r < g.W; ++r)
    for (int c = 0; c < g.D; ++c) {
      if (k) memcpy(k + r * g.D + c, buf.data() + qe::bf16_k_off(g, r, c), 2);
      if (v) memcpy(v + r * g.D + c, buf.data() + qe::bf16_v_off(g, r, c), 2);
    }
  return QE_OK;
}

qe_status qe_get_route_stats(qe_handle h, int layer, qe_route_stats* out) {
  if (h && h->tok) return fail(h, QE_ERR_STATE, "a window-tier call on a token-tiered handle");
  if (!h || !out) return QE_ERR_INVALID_ARG;
  if (layer < -1 || layer >= h->cfg.n_layers) return fail(h, QE_ERR_INVALID_ARG, "layer out of range");
  QE_CK(h, cudaStreamSynchronize(h->stream));
  std::vector<unsigned long long> v((size_t)h->cfg.n_layers * qe::N_STATS);
  QE_CK(h, cudaMemcpy(v.data(), h->st.stats, v.size() * 8, cudaMemcpyDeviceToHost));
  long long a[qe::N_STATS] = {};
  for (int l = 0; l < h->cfg.n_layers; ++l)
    if (layer == -1 || l == layer)
      for (int i = 0; i < qe::N_STATS; ++i) a[i] += (long long)v[(size_t)l * qe::N_STATS + i];
  out->routes = a[0];
  out->first_packs = a[1];
  out->ledger_reuses = a[2];
  out->promotions = a[3];
  out->evictions = a[4];
  out->bf16_reclaims = a[5];
  out->int2_reclaims = a[6];
  out->ledger_writes = a[7];
  return QE_OK;
}

qe_status qe_get_route_diag(qe_handle h, int layer, qe_route_diag* out, size_t n_units) {
  if (h && h->tok) return fail(h, QE_ERR_STATE, "a window-tier call on a token-tiered handle");
  if (!h || !out) return QE_ERR_INVALID_ARG;
  qe_status s = check_layer(h, layer);
  if (s != QE_OK) return s;
  if (n_units > (size_t)h->units) return fail(h, QE_ERR_INVALID_ARG, "n_units %zu > %d units", n_units, h->units);
  static_assert(sizeof(qe_route_diag) == sizeof(qe::RouteDiag), "routing record layout");
  QE_CK(h, cudaStreamSynchronize(h->stream));
  QE_CK(h, cudaMemcpy(out, h->diag + (size_t)layer * h->units, n_units * sizeof(qe_route_diag),
                      cudaMemcpyDeviceToHost));
  return QE_OK;
}

qe_status qe_debug_inject(qe_handle h, int what, long long value) {
  switch (what) {
    case QE_DEBUG_FAIL_DEVICE_ALLOC:
      if (value < 0) return QE_ERR_INVALID_ARG;
      g_fail_alloc_nth.store((int)value);
      return QE_OK;
    case QE_DEBUG_FAIL_HOST_STORE:
      g_fail_host_store.store(value != 0 ? 1 : 0);
      return QE_OK;
    case QE_DEBUG_EXPIRE_WAIT:
      if (!h) return QE_ERR_INVALID_ARG;
      if (value < 0 || value > (1 << 30)) return fail(h, QE_ERR_INVALID_ARG, "wait index %lld out of range", value);
      h->debug_expire = (int)value;
      return QE_OK;
    case QE_DEBUG_VERIFY_PATH:
      if (!h) return QE_ERR_INVALID_ARG;
      if (value < 0 || value > 2) return fail(h, QE_ERR_INVALID_ARG, "verify path %lld outside 0..2", value);
      h->verify_path = (int)value;
      return QE_OK;
    default:
      return h ? fail(h, QE_ERR_INVALID_ARG, "unknown injection %d", what) : QE_ERR_INVALID_ARG;
  }
}

qe_status qe_set_timing(qe_handle h, int enable) {
  if (!h) return QE_ERR_INVALID_ARG;
  h->timing = enable != 0;
  if (h->timing) {
    h->ev_used = 0;
    h->timed_bytes = 0;
    h->timed_launches = 0;
  }
  return QE_OK;
}

qe_status qe_launch_overhead(qe_handle h, int n, double* us) {
  if (!h || n < 1 || n > 10000 || !us) return h ? fail(h, QE_ERR_INVALID_ARG, "n %d or null output", n) : QE_ERR_INVALID_ARG;
  if (h->cfg.tiering != QE_TIERING_WINDOWS) return fail(h, QE_ERR_STATE, "window-tiered handles only");
  QE_CK(h, cudaStreamSynchronize(h->stream));
  QE_CK(h, qe::time_empty_attn_launch(h->cfg.head_dim, h->cfg.window, h->attn_grid, n, h->stream, us));
  return QE_OK;
}

qe_status qe_get_timing(qe_handle h, double* attn_ms, long long* launches, double* attn_bytes) {
  if (!h) return QE_ERR_INVALID_ARG;
  QE_CK(h, cudaStreamSynchronize(h->stream));
  double ms = 0;
  for (size_t i = 0; i + 1 < h->ev_used; i += 2) {
    float t = 0;
    QE_CK(h, cudaEventElapsedTime(&t, h->ev_pool[i], h->ev_pool[i + 1]));
    ms += t;
  }
  if (attn_ms) *attn_ms = ms;
  if (launches) *launches = h->timed_launches;
  if (attn_bytes) *attn_bytes = h->timed_bytes;
  return QE_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------------ snapshots
// The state a window-tiered handle carries from one call to the next: every device array of
// the table, the two slabs, the host store and ledger, the layer headers, the routing counters
// and records, and the host mirror of each layer.  Scratch (split-K partials, staging, move
// lists, verify deltas) is rebuilt by every call and not saved.
namespace {

struct Region {
  void* p;
  size_t bytes;
  bool host;   // pinned host memory (memcpy) rather than device memory (cudaMemcpy)
};

std::vector<Region> state_regions(qe_handle h) {
  const qe::State& st = h->st;
  const size_t GU = (size_t)h->gu_total, maxw = (size_t)st.maxw, capb = (size_t)st.capb, capq = (size_t)st.capq,
               caps = (size_t)st.caps, L = (size_t)h->cfg.n_layers;
  const size_t bslot_b = (size_t)st.geo.bslot_bytes(), qslot_b = (size_t)st.geo.qslot_bytes();
  return {
      {st.tier, GU * maxw, false},
      {st.bslot, GU * maxw * 4, false},
      {st.qslot, GU * maxw * 4, false},
      {st.sent, GU * maxw * 4, false},
      {st.score, GU * maxw * 4, false},
      {st.blist, GU * capb * sizeof(int2), false},
      {st.qlist, GU * capq * sizeof(int2), false},
      {st.bfree, GU * capb * 4, false},
      {st.bfree_head, GU * 4, false},
      {st.bfree_top, GU * 4, false},
      {st.bvictim, GU * capb * 4, false},
      {st.qvictim, GU * capq * 4, false},
      {st.bprev, GU * maxw * 4, false},
      {st.qprev, GU * maxw * 4, false},
      {st.qfree, GU * capq * 4, false},
      {st.qfree_top, GU * 4, false},
      {st.sfree, GU * caps * 4, false},
      {st.sfree_top, GU * 4, false},
      {st.bslab, GU * capb * bslot_b, false},
      {st.qslab, GU * capq * qslot_b, false},
      {st.qrange, GU * capq * 4, false},
      {st.err, 4, false},
      {st.stats, L * qe::N_STATS * sizeof(unsigned long long), false},
      {st.ldev, L * sizeof(qe::LayerDev), false},
      {h->diag, L * (size_t)h->units * sizeof(qe::RouteDiag), false},
      {h->hstore_host, GU * caps * bslot_b, true},
      {h->hledger_host, GU * caps * qslot_b, true},
  };
}

// The configuration fields that fix the layout, as doubles (no struct padding involved)
constexpr int SNAP_CFG = 22;
void snap_cfg(const qe_config& c, double (&v)[SNAP_CFG]) {
  const double x[SNAP_CFG] = {(double)c.batch, (double)c.n_layers, (double)c.n_q_heads, (double)c.n_kv_heads,
                              (double)c.head_dim, (double)c.window, (double)c.route_period, (double)c.n_sink,
                              (double)c.n_recent, (double)c.max_context, (double)c.cap_mode, (double)c.kf,
                              (double)c.kq, c.frac_bf16, c.frac_int2, c.budget_frac, (double)c.out_fp32,
                              (double)c.tiering, c.rope_theta, (double)c.int2_slack, c.frac_int4, c.frac_nq1};
  for (int i = 0; i < SNAP_CFG; ++i) v[i] = x[i];
}

constexpr char SNAP_MAGIC[8] = {'Q', 'E', 'S', 'N', 'A', 'P', '0', '1'};
struct SnapHeader {
  char magic[8];
  uint64_t total_bytes;
  uint64_t n_regions;
  double cfg[SNAP_CFG];
};
struct SnapLayer {
  int32_t L, routed_upto, n_full, n_quant, kf, kq;
};

size_t snap_bytes(qe_handle h, const std::vector<Region>& regs) {
  size_t n = sizeof(SnapHeader) + (size_t)h->cfg.n_layers * sizeof(SnapLayer) + regs.size() * sizeof(uint64_t);
  for (const Region& r : regs) n += r.bytes;
  return n;
}

qe_status snap_usable(qe_handle h) {
  if (!h) return QE_ERR_INVALID_ARG;
  if (h->tok) return fail(h, QE_ERR_STATE, "snapshots serve window-tiered handles");
  for (int l = 0; l < h->cfg.n_layers; ++l)
    if (h->lay[l].verify_n) return fail(h, QE_ERR_STATE, "layer %d awaits qe_verify_commit", l);
  return QE_OK;
}

}  // namespace

qe_status qe_snapshot_size(qe_handle h, size_t* bytes) {
  qe_status s = snap_usable(h);
  if (s != QE_OK) return s;
  if (!bytes) return fail(h, QE_ERR_INVALID_ARG, "bytes is null");
  *bytes = snap_bytes(h, state_regions(h));
  return QE_OK;
}

qe_status qe_snapshot(qe_handle h, void* host, size_t bytes) {
  qe::NvtxRange nvtx_("qe_snapshot");
  qe_status s = snap_usable(h);
  if (s != QE_OK) return s;
  const std::vector<Region> regs = state_regions(h);
  const size_t need = snap_bytes(h, regs);
  if (!host || bytes < need) return fail(h, QE_ERR_INVALID_ARG, "snapshot needs %zu bytes", need);
  for (int l = 0; l < h->cfg.n_layers; ++l)   // a pending single-token append is written first
    if ((s = commit_pending(h, l)) != QE_OK) return s;
  QE_CK(h, cudaStreamSynchronize(h->stream));
  uint8_t* o = static_cast<uint8_t*>(host);
  SnapHeader hd{};
  std::memcpy(hd.magic, SNAP_MAGIC, 8);
  hd.total_bytes = need;
  hd.n_regions = regs.size();
  snap_cfg(h->cfg, hd.cfg);
  std::memcpy(o, &hd, sizeof hd);
  o += sizeof hd;
  for (int l = 0; l < h->cfg.n_layers; ++l) {
    const LayerMirror& m = h->lay[l];
    const SnapLayer sl{m.L, m.routed_upto, m.n_full, m.n_quant, m.kf, m.kq};
    std::memcpy(o, &sl, sizeof sl);
    o += sizeof sl;
  }
  for (const Region& r : regs) {
    const uint64_t b = r.bytes;
    std::memcpy(o, &b, sizeof b);
    o += sizeof b;
  }
  for (const Region& r : regs) {
    if (r.host) std::memcpy(o, r.p, r.bytes);
    else QE_CK(h, cudaMemcpy(o, r.p, r.bytes, cudaMemcpyDeviceToHost));
    o += r.bytes;
  }
  return QE_OK;
}

qe_status qe_restore(qe_handle h, const void* host, size_t bytes) {
  qe::NvtxRange nvtx_("qe_restore");
  qe_status s = snap_usable(h);
  if (s != QE_OK) return s;
  const std::vector<Region> regs = state_regions(h);
  const size_t need = snap_bytes(h, regs);
  if (!host || bytes < sizeof(SnapHeader)) return fail(h, QE_ERR_INVALID_ARG, "not a snapshot");
  const uint8_t* in = static_cast<const uint8_t*>(host);
  SnapHeader hd;
  std::memcpy(&hd, in, sizeof hd);
  if (std::memcmp(hd.magic, SNAP_MAGIC, 8) != 0) return fail(h, QE_ERR_INVALID_ARG, "not a snapshot");
  double cfg[SNAP_CFG];
  snap_cfg(h->cfg, cfg);
  for (int i = 0; i < SNAP_CFG; ++i)
    if (cfg[i] != hd.cfg[i]) return fail(h, QE_ERR_INVALID_ARG, "snapshot of another configuration (field %d)", i);
  if (hd.total_bytes != need || bytes < need || hd.n_regions != regs.size())
    return fail(h, QE_ERR_INVALID_ARG, "snapshot of %llu bytes, this handle's are %zu",
                (unsigned long long)hd.total_bytes, need);
  const uint8_t* p = in + sizeof hd;
  std::vector<SnapLayer> lays((size_t)h->cfg.n_layers);
  for (int l = 0; l < h->cfg.n_layers; ++l) {
    std::memcpy(&lays[(size_t)l], p, sizeof(SnapLayer));
    p += sizeof(SnapLayer);
  }
  for (const Region& r : regs) {
    uint64_t b;
    std::memcpy(&b, p, sizeof b);
    p += sizeof b;
    if (b != r.bytes) return fail(h, QE_ERR_INVALID_ARG, "snapshot region of %llu bytes, expected %zu",
                                  (unsigned long long)b, r.bytes);
  }
  // the handle's own work is finished before its state is replaced
  QE_CK(h, cudaStreamSynchronize(h->stream));
  for (const Region& r : regs) {
    if (r.host) std::memcpy(r.p, p, r.bytes);
    else QE_CK(h, cudaMemcpy(r.p, p, r.bytes, cudaMemcpyHostToDevice));
    p += r.bytes;
  }
  for (int l = 0; l < h->cfg.n_layers; ++l) {
    LayerMirror m{};
    const SnapLayer& sl = lays[(size_t)l];
    m.L = sl.L;
    m.routed_upto = sl.routed_upto;
    m.n_full = sl.n_full;
    m.n_quant = sl.n_quant;
    m.kf = sl.kf;
    m.kq = sl.kq;
    h->lay[(size_t)l] = m;
  }
  return QE_OK;
}
