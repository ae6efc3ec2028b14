// qe_tok_host.cu -- host side of the five-tier per-token cache (QE_TIERING_TOKENS): handle set-up,
// launches behind qe_append / qe_decode_step / qe_route, and the introspection calls.
//
// Per-unit tier counts change only at a re-rank and live on the device; the host keeps the
// length, the tail count and the pending token of every layer (all units share them).
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "qe.h"
#include "qe_handle.hpp"
#include "qe_tok_kernels.h"

namespace qe {
namespace {

qe_status tfail(qe_handle h, qe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  h->err = buf;
  return s;
}

#define TK_CK(h, call)                                                                               \
  do {                                                                                               \
    cudaError_t e_ = (call);                                                                         \
    if (e_ != cudaSuccess)                                                                           \
      return tfail((h), e_ == cudaErrorMemoryAllocation ? QE_ERR_OOM : QE_ERR_CUDA, "%s: %s (%s:%d)", \
                   #call, cudaGetErrorString(e_), __FILE__, __LINE__);                               \
  } while (0)

int round16(long long x) { return (int)((x + 15) / 16 * 16); }

template <class T>
cudaError_t talloc(qe_handle h, T** p, size_t count) {
  void* q = nullptr;
  if (inject_alloc_failure()) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(&q, count > 0 ? count * sizeof(T) : 16);
  if (e != cudaSuccess) return e;
  h->tk_allocs.push_back(q);
  *p = static_cast<T*>(q);
  return cudaMemsetAsync(q, 0, count > 0 ? count * sizeof(T) : 16, h->stream);
}

// device view of a pinned, mapped host buffer (nullptr for pageable memory)
const void* mapped(const void* p, size_t align) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  if (reinterpret_cast<uintptr_t>(a.devicePointer) % align) return nullptr;
  return a.devicePointer;
}

qe_status stage(qe_handle h, int i, size_t bytes, void** out) {
  if (h->stage_bytes[i] < bytes) {
    if (h->stage[i]) cudaFree(h->stage[i]);
    h->stage[i] = nullptr;
    h->stage_bytes[i] = 0;
    TK_CK(h, cudaMalloc(&h->stage[i], bytes));
    h->stage_bytes[i] = bytes;
  }
  *out = h->stage[i];
  return QE_OK;
}

qe_status check(qe_handle h, int layer) {
  if (layer < 0 || layer >= h->cfg.n_layers) return tfail(h, QE_ERR_INVALID_ARG, "layer %d out of range", layer);
  return QE_OK;
}

// Writes the pending token into the tail if no decode step has written it yet.
qe_status flush_token(qe_handle h, int layer) {
  TokMirror& m = h->tlay[layer];
  if (!m.pk) return QE_OK;
  TK_CK(h, tk_launch_append1(h->ts, layer, m.pk, m.pv, h->stream));
  ++h->launches;
  m.pk = m.pv = nullptr;
  return QE_OK;
}

qe_status commit(qe_handle h, int layer) {
  TokMirror& m = h->tlay[layer];
  if (!m.pending) return QE_OK;
  qe_status st = flush_token(h, layer);
  if (st != QE_OK) return st;
  TK_CK(h, tk_launch_commit_pending(h->ts, layer, m.pending, h->stream));
  ++h->launches;
  m.pending = 0;
  return QE_OK;
}

// Algorithmic bytes one attention launch reads: BF16 tokens 4 d, b-bit tokens 2 (d b / 8 + 8).
double attn_bytes(qe_handle h, const std::vector<int>& cnt, int n_tail) {
  const int D = h->cfg.head_dim;
  double b = 0;
  for (int u = 0; u < h->ts.units; ++u) {
    b += (double)(cnt[u * 4 + 0] + n_tail) * 4.0 * D;
    b += (double)cnt[u * 4 + 1] * 2.0 * (D * 4 / 8 + 8);
    b += (double)cnt[u * 4 + 2] * 2.0 * (D * 2 / 8 + 8);
    b += (double)cnt[u * 4 + 3] * 2.0 * (D * 1 / 8 + 8);
  }
  return b;
}

qe_status fetch_counts(qe_handle h, int layer, std::vector<int>& cnt, TokLayer& hd) {
  cnt.assign((size_t)h->ts.units * 4, 0);
  TK_CK(h, cudaStreamSynchronize(h->stream));
  TK_CK(h, cudaMemcpy(cnt.data(), h->ts.cnt + (size_t)layer * h->ts.units * 4, cnt.size() * 4, cudaMemcpyDeviceToHost));
  TK_CK(h, cudaMemcpy(&hd, h->ts.hdr + layer, sizeof(TokLayer), cudaMemcpyDeviceToHost));
  return QE_OK;
}

}  // namespace

qe_status tok_init(const qe_config& c, cudaStream_t stream, qe_handle* out, std::string& err) {
  const int G = c.n_q_heads / c.n_kv_heads;
  const double f[4] = {c.frac_bf16, c.frac_int4, c.frac_int2, c.frac_nq1};
  for (double x : f)
    if (!(x >= 0.0 && x <= 1.0)) {
      err = "token fractions must be in [0, 1]";
      return QE_ERR_INVALID_ARG;
    }
  if (f[0] + f[1] + f[2] + f[3] > 1.0 + 1e-12) {
    err = "token fractions must sum to at most 1";
    return QE_ERR_INVALID_ARG;
  }
  if (c.route_period < 1 || c.score_window < 0 || c.score_window > c.route_period) {
    err = "need route_period >= 1 and 0 <= score_window <= route_period";
    return QE_ERR_INVALID_ARG;
  }
  if (c.n_sink < 0 || c.n_recent < 1) {
    err = "need n_sink >= 0 and n_recent >= 1";
    return QE_ERR_INVALID_ARG;
  }
  qe_handle h = new qe_handle_s();
  h->cfg = c;
  h->stream = stream;
  h->tok = true;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    delete h;
    err = std::string("no CUDA device: ") + cudaGetErrorString(e);
    return QE_ERR_CUDA;
  }
  TokState& s = h->ts;
  s.g.D = c.head_dim;
  s.units = c.batch * c.n_kv_heads;
  s.G = G;
  s.Hkv = c.n_kv_heads;
  s.Hq = c.n_q_heads;
  s.n_sink = c.n_sink;
  s.n_recent = c.n_recent;
  s.max_context = c.max_context;
  s.period = c.route_period;
  s.score_window = c.score_window;
  for (int z = 0; z < 4; ++z) s.frac[z] = f[z];
  // a pool's count never exceeds the cumulative fraction of L (demote only), except the BF16
  // pool, which holds the prefill until the first re-rank
  s.cap[0] = round16(c.max_context);
  double cf = f[0];
  for (int z = 1; z < 4; ++z) {
    cf += f[z];
    long long n = (long long)std::floor(cf * c.max_context) + 1;
    if (n > c.max_context) n = c.max_context;
    s.cap[z] = round16(n);
  }
  s.cap_tail = round16((long long)c.n_sink + c.n_recent + 2LL * c.route_period + 16);
  s.cost[0] = 8; s.cost[1] = 4; s.cost[2] = 3; s.cost[3] = 3; s.cost[4] = 8;
  h->units = s.units;
  h->tlay.assign(c.n_layers, TokMirror{});
  const long long LB = 2LL * c.n_layers * s.units;   // layers x buffers x units
  const size_t mc = (size_t)c.max_context;
  h->tk_grid = h->n_sm;
  const int NW = h->tk_grid * tk_attn_warps();
  h->tk_lgcap = s.cap[0] + s.cap[1] + s.cap[2] + s.cap[3] + s.cap_tail;
  cudaError_t ae = cudaSuccess;
  auto A = [&](cudaError_t x) { if (ae == cudaSuccess) ae = x; };
  for (int z = 0; z < 4; ++z) {
    A(talloc(h, &s.pool[z], (size_t)LB * (s.cap[z] / 16) * tk_tile_bytes(s, z)));
    A(talloc(h, &s.pos[z], (size_t)LB * s.cap[z]));
    A(talloc(h, &s.score[z], (size_t)LB * s.cap[z]));
  }
  A(talloc(h, &s.tail, (size_t)LB * (s.cap_tail / 16) * s.g.bf_tile()));
  A(talloc(h, &s.tail_pos, (size_t)LB * s.cap_tail));
  A(talloc(h, &s.tail_score, (size_t)LB * s.cap_tail));
  A(talloc(h, &s.hdr, (size_t)c.n_layers));
  A(talloc(h, &s.cnt, (size_t)c.n_layers * s.units * 4));
  A(talloc(h, &s.cum, (size_t)c.n_layers * (s.units + 1)));
  A(talloc(h, &s.err, 1));
  // re-rank scratch, one slot per layer: qe_route(-1) re-ranks every layer in one launch
  const size_t NLU = (size_t)c.n_layers * s.units;
  A(talloc(h, &s.ckey, NLU * mc));
  A(talloc(h, &s.csrc, NLU * mc));
  A(talloc(h, &s.newt, NLU * mc));
  A(talloc(h, &s.order, NLU * 4 * mc));
  A(talloc(h, &s.src_of, NLU * mc));
  A(talloc(h, &s.ncnt, NLU * 4));
  A(talloc(h, &s.done, (size_t)c.n_layers));
  A(talloc(h, &h->tk_part_o, (size_t)(NW + s.units) * G * c.head_dim));
  A(talloc(h, &h->tk_part_ml, (size_t)(NW + s.units) * G));
  A(talloc(h, &h->tk_logits, (size_t)s.units * h->tk_lgcap * G));
  A(talloc(h, &h->tok_stage, (size_t)c.n_layers * 2 * s.units * c.head_dim));
  A(tk_prepare(c.head_dim));
  A(cudaStreamSynchronize(stream));
  if (ae != cudaSuccess) {
    err = std::string("setting up the five-tier cache: ") + cudaGetErrorString(ae) + injected_note();
    tok_free(h);
    delete h;
    return ae == cudaErrorMemoryAllocation ? QE_ERR_OOM : QE_ERR_CUDA;
  }
  h->st.err = s.err;   // qe_synchronize reads the sticky flag here
  *out = h;
  return QE_OK;
}

void tok_free(qe_handle h) {
  for (void* p : h->tk_allocs) cudaFree(p);
  h->tk_allocs.clear();
  for (int i = 0; i < 4; ++i)
    if (h->stage[i]) cudaFree(h->stage[i]);
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  h->ev_pool.clear();
  h->st.err = nullptr;
}

qe_status tok_append(qe_handle h, int layer, const void* k, const void* v, int n, int flags) {
  qe_status st = check(h, layer);
  if (st != QE_OK) return st;
  if (!k || !v || n < 1) return tfail(h, QE_ERR_INVALID_ARG, "append needs K, V and n_tokens >= 1");
  TokMirror& m = h->tlay[layer];
  const TokState& s = h->ts;
  if (m.L + n > h->cfg.max_context)
    return tfail(h, QE_ERR_CAPACITY, "append of %d tokens passes max_context %d (length %d)", n, h->cfg.max_context, m.L);
  const bool prefill = m.L == 0 && n > 1;
  int tail_after;
  if (prefill) {
    const int lo = s.n_sink < n ? s.n_sink : n;
    const int hi = n - s.n_recent > lo ? n - s.n_recent : lo;
    tail_after = lo + (n - hi);
  } else {
    tail_after = m.n_tail + n;
  }
  if (tail_after > s.cap_tail)
    return tfail(h, QE_ERR_CAPACITY, "the BF16 tail holds %d tokens: re-rank (qe_route) at least every route_period steps",
                 s.cap_tail);
  if ((st = commit(h, layer)) != QE_OK) return st;
  const size_t bytes = (size_t)s.units * n * h->cfg.head_dim * 2;
  const uint16_t* kd = static_cast<const uint16_t*>(k);
  const uint16_t* vd = static_cast<const uint16_t*>(v);
  if (n == 1) {
    // The token is written by the next decode step's attention launch (or by a launch of its
    // own before any other call reads the layer).  Host memory: pinned is read in place,
    // pageable is copied now into this layer's staging.
    if (flags & QE_HOST_PTRS) {
      const void* mk = mapped(k, 4);
      const void* mv = mapped(v, 2);
      if (mk && mv) {
        kd = static_cast<const uint16_t*>(mk);
        vd = static_cast<const uint16_t*>(mv);
      } else {
        uint16_t* ks = h->tok_stage + (size_t)layer * 2 * s.units * h->cfg.head_dim;
        uint16_t* vs = ks + (size_t)s.units * h->cfg.head_dim;
        TK_CK(h, cudaMemcpyAsync(ks, k, bytes, cudaMemcpyHostToDevice, h->stream));
        TK_CK(h, cudaMemcpyAsync(vs, v, bytes, cudaMemcpyHostToDevice, h->stream));
        kd = ks;
        vd = vs;
      }
    }
    m.pk = kd;
    m.pv = vd;
    m.pending = 1;
    m.L += 1;
    m.n_tail += 1;
    return QE_OK;
  }
  if (flags & QE_HOST_PTRS) {
    void *sk, *sv;
    if ((st = stage(h, 0, bytes, &sk)) != QE_OK || (st = stage(h, 1, bytes, &sv)) != QE_OK) return st;
    TK_CK(h, cudaMemcpyAsync(sk, k, bytes, cudaMemcpyHostToDevice, h->stream));
    TK_CK(h, cudaMemcpyAsync(sv, v, bytes, cudaMemcpyHostToDevice, h->stream));
    kd = static_cast<const uint16_t*>(sk);
    vd = static_cast<const uint16_t*>(sv);
  }
  TK_CK(h, tk_launch_append(s, layer, n, prefill, kd, vd, h->n_sm, h->stream));
  h->launches += 2;
  m.L += n;
  m.n_tail = tail_after;
  return QE_OK;
}

qe_status tok_decode(qe_handle h, int layer, const void* q, void* out, int flags) {
  qe_status st = check(h, layer);
  if (st != QE_OK) return st;
  if (!q || !out) return tfail(h, QE_ERR_INVALID_ARG, "decode needs q and out");
  TokMirror& m = h->tlay[layer];
  if (m.L < 1) return tfail(h, QE_ERR_STATE, "decode on an empty layer");
  const qe_config& c = h->cfg;
  const int D = c.head_dim;
  const size_t qbytes = (size_t)c.batch * c.n_q_heads * D * 2;
  const size_t obytes = (size_t)c.batch * c.n_q_heads * D * (c.out_fp32 ? 4 : 2);
  const uint16_t* qd = static_cast<const uint16_t*>(q);
  void* od = out;
  bool out_copy = false;
  if (flags & QE_HOST_PTRS) {
    if (const void* mq = mapped(q, 4)) {
      qd = static_cast<const uint16_t*>(mq);
    } else {
      void* sq;
      if ((st = stage(h, 2, qbytes, &sq)) != QE_OK) return st;
      TK_CK(h, cudaMemcpyAsync(sq, q, qbytes, cudaMemcpyHostToDevice, h->stream));
      qd = static_cast<const uint16_t*>(sq);
    }
    if (const void* mo = mapped(out, c.out_fp32 ? 4 : 2)) {
      od = const_cast<void*>(mo);
    } else {
      if ((st = stage(h, 3, obytes, &od)) != QE_OK) return st;
      out_copy = true;
    }
  }
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  unsigned ev_flags = cudaEventRecordDefault;
  if (h->timing) {
    while (h->ev_pool.size() < h->ev_used + 2) {
      cudaEvent_t ev;
      TK_CK(h, cudaEventCreate(&ev));
      h->ev_pool.push_back(ev);
    }
    e0 = h->ev_pool[h->ev_used];
    e1 = h->ev_pool[h->ev_used + 1];
    h->ev_used += 2;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    TK_CK(h, cudaStreamIsCapturing(h->stream, &cs));
    ev_flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    TK_CK(h, cudaEventRecordWithFlags(e0, h->stream, ev_flags));
  }
  TK_CK(h, tk_launch_attn(h->ts, layer, m.pending, m.pk, m.pv, qd, scale_log2, h->tk_part_o, h->tk_part_ml,
                          h->tk_logits, h->tk_lgcap, h->tk_grid, h->stream, h->debug_expire));
  h->debug_expire = 0;   // one step only
  ++h->launches;
  m.pk = m.pv = nullptr;   // written by this launch
  if (h->timing) {
    TK_CK(h, cudaEventRecordWithFlags(e1, h->stream, ev_flags));
    h->timed_launches += 1;
    std::vector<int> cnt;
    TokLayer hd;
    qe_status fs = fetch_counts(h, layer, cnt, hd);   // synchronising: timing mode only
    if (fs != QE_OK) return fs;
    h->timed_bytes += attn_bytes(h, cnt, m.n_tail);
  }
  TK_CK(h, tk_launch_merge(h->ts, layer, m.pending, h->tk_part_o, h->tk_part_ml, h->tk_logits, h->tk_lgcap,
                           h->tk_grid, od, c.out_fp32, h->stream));
  ++h->launches;
  m.pending = 0;
  if (out_copy) TK_CK(h, cudaMemcpyAsync(out, od, obytes, cudaMemcpyDeviceToHost, h->stream));
  return QE_OK;
}

qe_status tok_route(qe_handle h, int layer) {
  const int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? h->cfg.n_layers : layer + 1;
  if (layer >= h->cfg.n_layers) return tfail(h, QE_ERR_INVALID_ARG, "layer %d out of range", layer);
  for (int l = l0; l < l1; ++l) {
    qe_status st = commit(h, l);
    if (st != QE_OK) return st;
  }
  TK_CK(h, tk_launch_rerank(h->ts, l0, l1 - l0, h->stream));
  h->launches += 3;
  for (int l = l0; l < l1; ++l) {
    TokMirror& m = h->tlay[l];
    int aged = m.n_tail - h->ts.n_sink - h->ts.n_recent;
    if (aged < 0) aged = 0;
    m.n_tail -= aged;
  }
  return QE_OK;
}

qe_status tok_layer_info(qe_handle h, int layer, qe_layer_info* info) {
  qe_status st = check(h, layer);
  if (st != QE_OK) return st;
  std::vector<int> cnt;
  TokLayer hd;
  if ((st = fetch_counts(h, layer, cnt, hd)) != QE_OK) return st;
  std::memset(info, 0, sizeof *info);
  TokMirror& m = h->tlay[layer];
  m.L = hd.L + m.pending;              // the device header also advances under CUDA-graph replays
  m.n_tail = hd.n_tail + m.pending;
  info->length = m.L;
  info->units = h->ts.units;
  info->max_windows = h->cfg.max_context;
  info->attn_bytes = attn_bytes(h, cnt, m.n_tail);
  return QE_OK;
}

}  // namespace qe

// ------------------------------------------------------------------------------ introspection
extern "C" {

static qe_status tok_only(qe_handle h, int layer) {
  if (!h) return QE_ERR_INVALID_ARG;
  if (!h->tok) {
    h->err = "a five-tier call on a window-tiered handle";
    return QE_ERR_STATE;
  }
  if (layer < 0 || layer >= h->cfg.n_layers) {
    h->err = "layer out of range";
    return QE_ERR_INVALID_ARG;
  }
  return QE_OK;
}

// positions of every pool and of the tail, current buffer, all units; tier, index per token
struct TokSnapshot {
  std::vector<int> cnt;
  qe::TokLayer hd;
  std::vector<int> pos[5];
  std::vector<float> sc[5];
};

static qe_status tok_snapshot(qe_handle h, int layer, TokSnapshot& sn, bool scores) {
  const qe::TokState& s = h->ts;
  qe_status fs = qe::flush_token(h, layer);   // the pending token is read from the tail below
  if (fs != QE_OK) return fs;
  sn.cnt.assign((size_t)s.units * 4, 0);
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e == cudaSuccess)
    e = cudaMemcpy(sn.cnt.data(), s.cnt + (size_t)layer * s.units * 4, sn.cnt.size() * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&sn.hd, s.hdr + layer, sizeof sn.hd, cudaMemcpyDeviceToHost);
  for (int z = 0; z < 5 && e == cudaSuccess; ++z) {
    const int cap = z < 4 ? s.cap[z] : s.cap_tail;
    const long long base = z < 4 ? qe::tk_pool_tok_index(s, z, layer, sn.hd.buf, 0) : qe::tk_tail_tok_index(s, layer, sn.hd.buf, 0);
    sn.pos[z].assign((size_t)s.units * cap, 0);
    e = cudaMemcpy(sn.pos[z].data(), (z < 4 ? s.pos[z] : s.tail_pos) + base, sn.pos[z].size() * 4, cudaMemcpyDeviceToHost);
    if (scores && e == cudaSuccess) {
      sn.sc[z].assign((size_t)s.units * cap, 0.f);
      e = cudaMemcpy(sn.sc[z].data(), (z < 4 ? s.score[z] : s.tail_score) + base, sn.sc[z].size() * 4,
                     cudaMemcpyDeviceToHost);
    }
  }
  if (e != cudaSuccess) {
    h->err = std::string("reading the five-tier cache: ") + cudaGetErrorString(e);
    return QE_ERR_CUDA;
  }
  return QE_OK;
}

static int tok_count(const qe_handle h, const TokSnapshot& sn, int layer, int u, int z) {
  if (z < 4) return sn.cnt[(size_t)u * 4 + z];
  return sn.hd.n_tail + h->tlay[layer].pending;   // the pending token is written already
}
static int tok_length(const qe_handle h, const TokSnapshot& sn, int layer) { return sn.hd.L + h->tlay[layer].pending; }

qe_status qe_get_token_tiers(qe_handle h, int layer, uint8_t* host, size_t bytes) {
  qe_status st = tok_only(h, layer);
  if (st != QE_OK) return st;
  const qe::TokState& s = h->ts;
  const size_t mc = (size_t)s.max_context;
  if (!host || bytes < (size_t)s.units * mc) {
    h->err = "token tier buffer too small";
    return QE_ERR_INVALID_ARG;
  }
  TokSnapshot sn;
  if ((st = tok_snapshot(h, layer, sn, false)) != QE_OK) return st;
  const int L = tok_length(h, sn, layer);
  for (int u = 0; u < s.units; ++u) {
    uint8_t* row = host + u * mc;
    for (size_t p = 0; p < mc; ++p) row[p] = (int)p < L ? QE_TOK_EVICTED : QE_TOK_ABSENT;
    for (int z = 0; z < 5; ++z) {
      const int cap = z < 4 ? s.cap[z] : s.cap_tail;
      const int n = tok_count(h, sn, layer, u, z);
      for (int i = 0; i < n; ++i) {
        const int p = sn.pos[z][(size_t)u * cap + i];
        if (p >= 0 && (size_t)p < mc) row[p] = (uint8_t)(z < 4 ? z : QE_TOK_BF16);
      }
    }
  }
  return QE_OK;
}

qe_status qe_get_token_scores(qe_handle h, int layer, float* host, size_t bytes) {
  qe_status st = tok_only(h, layer);
  if (st != QE_OK) return st;
  const qe::TokState& s = h->ts;
  const size_t mc = (size_t)s.max_context;
  if (!host || bytes < (size_t)s.units * mc * 4) {
    h->err = "token score buffer too small";
    return QE_ERR_INVALID_ARG;
  }
  TokSnapshot sn;
  if ((st = tok_snapshot(h, layer, sn, true)) != QE_OK) return st;
  for (int u = 0; u < s.units; ++u) {
    float* row = host + u * mc;
    for (size_t p = 0; p < mc; ++p) row[p] = 0.f;
    for (int z = 0; z < 5; ++z) {
      const int cap = z < 4 ? s.cap[z] : s.cap_tail;
      const int n = tok_count(h, sn, layer, u, z);
      for (int i = 0; i < n; ++i) {
        const int p = sn.pos[z][(size_t)u * cap + i];
        if (p >= 0 && (size_t)p < mc) row[p] = sn.sc[z][(size_t)u * cap + i];
      }
    }
  }
  return QE_OK;
}

qe_status qe_get_token_counts(qe_handle h, int layer, int* host, size_t bytes) {
  qe_status st = tok_only(h, layer);
  if (st != QE_OK) return st;
  const qe::TokState& s = h->ts;
  if (!host || bytes < (size_t)s.units * 5 * 4) {
    h->err = "token count buffer too small";
    return QE_ERR_INVALID_ARG;
  }
  TokSnapshot sn;
  if ((st = tok_snapshot(h, layer, sn, false)) != QE_OK) return st;
  for (int u = 0; u < s.units; ++u)
    for (int z = 0; z < 5; ++z) host[u * 5 + z] = tok_count(h, sn, layer, u, z);
  return QE_OK;
}

qe_status qe_get_token(qe_handle h, int layer, int unit, int pos, int* tier, uint16_t* k_bf16, uint16_t* v_bf16,
                       uint8_t* k_codes, uint8_t* v_codes, float* params) {
  qe_status st = tok_only(h, layer);
  if (st != QE_OK) return st;
  const qe::TokState& s = h->ts;
  if (unit < 0 || unit >= s.units || !tier) {
    h->err = "bad unit or null tier";
    return QE_ERR_INVALID_ARG;
  }
  TokSnapshot sn;
  if ((st = tok_snapshot(h, layer, sn, false)) != QE_OK) return st;
  *tier = pos >= 0 && pos < tok_length(h, sn, layer) ? QE_TOK_EVICTED : QE_TOK_ABSENT;
  const int D = s.g.D;
  for (int z = 0; z < 5; ++z) {
    const int cap = z < 4 ? s.cap[z] : s.cap_tail;
    const int n = tok_count(h, sn, layer, unit, z);
    for (int i = 0; i < n; ++i) {
      if (sn.pos[z][(size_t)unit * cap + i] != pos) continue;
      const int zz = z < 4 ? z : qe::TK_TAIL;
      const uint8_t* dev = z < 4 ? s.pool[z] + (qe::tk_pool_tile_index(s, z, layer, sn.hd.buf, unit) + i / 16) *
                                                   (long long)qe::tk_tile_bytes(s, z)
                                 : s.tail + (qe::tk_tail_tok_index(s, layer, sn.hd.buf, unit) / 16 + i / 16) *
                                                (long long)s.g.bf_tile();
      std::vector<uint8_t> tile((size_t)qe::tk_tile_bytes(s, zz));
      if (cudaMemcpy(tile.data(), dev, tile.size(), cudaMemcpyDeviceToHost) != cudaSuccess) {
        h->err = "reading a tile";
        return QE_ERR_CUDA;
      }
      const int row = i & 15;
      if (zz == qe::TK_BF16 || zz == qe::TK_TAIL) {
        *tier = QE_TOK_BF16;
        const qe::Geo g16{D, 16};
        for (int c = 0; c < D; ++c) {
          if (k_bf16) std::memcpy(k_bf16 + c, tile.data() + qe::bf16_k_off(g16, row, c), 2);
          if (v_bf16) std::memcpy(v_bf16 + c, tile.data() + qe::bf16_v_off(g16, row, c), 2);
        }
        return QE_OK;
      }
      *tier = z;
      const int b = qe::tk_bits(z);
      for (int c = 0; c < D; ++c) {
        for (int val = 0; val < 2; ++val) {
          const qe::CodePos cp = val ? qe::tk_vcode_pos(s.g, b, row, c) : qe::tk_kcode_pos(s.g, b, row, c);
          unsigned w;
          std::memcpy(&w, tile.data() + cp.byte, 4);
          const uint8_t code = (uint8_t)((w >> cp.bit) & ((1u << b) - 1u));
          uint8_t* dst = val ? v_codes : k_codes;
          if (dst) dst[c] = code;
        }
      }
      if (params) {
        std::memcpy(params + 0, tile.data() + s.g.off_kpar(b) + row * 8, 8);
        std::memcpy(params + 2, tile.data() + s.g.off_vpar(b) + row * 8, 8);
      }
      return QE_OK;
    }
  }
  return QE_OK;
}

}  // extern "C"
