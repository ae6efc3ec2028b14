// qe_noalloc.cu -- qe_decode_step_noalloc: one decode step that allocates no device memory.
//
// Who needs it.  Some callers run the decode path where they may not call cudaMalloc: code
// whose device memory is owned by an arena or budget manager that forbids new allocations
// once serving has started, code running where a cudaMalloc could block on the allocator or
// synchronise the device at the wrong moment, or code on a thread that is not allowed to make
// allocating CUDA calls at all.  qe_decode_step itself allocates nothing per call once its
// handle exists, except the staging buffers it creates on first use for host pointers; this
// entry point accepts device pointers only and takes the split-K scratch of the attention
// (per-warp partial outputs and per-tile log-sum-exps) from a
// fixed array compiled into the library instead of the handle's own scratch.  The kernels are
// the same two the handle's decode step launches.
//
// The array is a file-scope static __device__ variable: every GPU that loads the library keeps
// NA_BYTES (about 4.1 MiB) reserved until the process exits.  In host code its name is only a
// host-side stand-in, so its device address is looked up with cudaGetSymbolAddress on the
// first call on each device (with that device current) and cached.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include <cuda_runtime.h>

#include "qe.h"
#include "qe_handle.hpp"
#include "qe_kernels.cuh"

namespace {

constexpr int NA_MAX_UNITS = 16;       // batch * n_kv_heads
constexpr int NA_PSLOTS = 64;          // split-K partial slots per unit
constexpr int NA_MAX_TILES = 8192;     // 16-token bf16 sub-tiles + 2-bit windows per unit
constexpr int NA_MAX_G = 4;
constexpr int NA_MAX_D = 128;
constexpr size_t NA_PART_O = (size_t)NA_MAX_UNITS * NA_PSLOTS * NA_MAX_G * NA_MAX_D * sizeof(float);
constexpr size_t NA_PART_ML = (size_t)NA_MAX_UNITS * NA_PSLOTS * NA_MAX_G * sizeof(float2);
constexpr size_t NA_LSE = (size_t)NA_MAX_UNITS * NA_MAX_TILES * NA_MAX_G * sizeof(float);
constexpr size_t NA_BYTES = NA_PART_O + NA_PART_ML + NA_LSE;

static __device__ __align__(256) unsigned char g_na_scratch[NA_BYTES];

constexpr int NA_MAX_DEVICES = 128;
std::mutex g_na_mu;
void* g_na_ptr[NA_MAX_DEVICES] = {};

qe_status na_fail(qe_handle h, qe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  h->err = buf;
  return s;
}

}  // namespace

extern "C" qe_status qe_decode_step_noalloc(qe_handle h, int layer, const void* q, void* out) {
  qe::NvtxRange nvtx_("qe_decode_step_noalloc");
  if (!h) return QE_ERR_INVALID_ARG;
  if (h->tok) return na_fail(h, QE_ERR_STATE, "the no-allocation decode step serves window-tiered handles");
  if (layer < 0 || layer >= h->cfg.n_layers) return na_fail(h, QE_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (!q || !out) return na_fail(h, QE_ERR_INVALID_ARG, "noalloc decode needs device q and out");
  qe::LayerMirror& m = h->lay[layer];
  // a speculative verify leaves uncommitted drafts in the layer: attending over them here would
  // add their masses to the scores, which the commit could not take back
  if (m.verify_n) return na_fail(h, QE_ERR_STATE, "layer %d awaits qe_verify_commit", layer);
  if (m.L < 1) return na_fail(h, QE_ERR_STATE, "decode on an empty layer");
  const int W = h->cfg.window, D = h->cfg.head_dim, G = h->st.G;
  if (h->units > NA_MAX_UNITS)
    return na_fail(h, QE_ERR_CAPACITY, "noalloc decode supports at most %d units (batch x KV heads), handle has %d",
                   NA_MAX_UNITS, h->units);
  const int nwin = (m.L + W - 1) / W;
  const int nbw = 1 + m.n_full + (nwin - m.routed_upto);
  const int ntiles = nbw * (W / 16) + m.n_quant;
  if (ntiles > NA_MAX_TILES)
    return na_fail(h, QE_ERR_CAPACITY, "noalloc decode supports at most %d tiles per unit, layer has %d",
                   NA_MAX_TILES, ntiles);
  if (G > NA_MAX_G || D > NA_MAX_D) return na_fail(h, QE_ERR_CAPACITY, "noalloc decode: head shape too large");

  // Device address of the static scratch on the handle's device (looked up once per device).
  // The kernels run on the handle's stream, which belongs to the device the handle was created
  // on; the array's address is only valid there, so that device must be the current one.
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return na_fail(h, QE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev != h->device)
    return na_fail(h, QE_ERR_STATE, "the current device %d is not the handle's device %d", dev, h->device);
  if (dev < 0 || dev >= NA_MAX_DEVICES) return na_fail(h, QE_ERR_INVALID_ARG, "device %d out of range", dev);
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (!g_na_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_na_scratch);
      if (e != cudaSuccess || !p)
        return na_fail(h, QE_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
      g_na_ptr[dev] = p;
    }
    base = static_cast<unsigned char*>(g_na_ptr[dev]);
  }
  // Nothing in the scratch has to start at zero: every partial slot a unit's combine reads and
  // every tile's log-sum-exp are written by this call's attention launch before they are read.
  float* part_o = reinterpret_cast<float*>(base);
  float2* part_ml = reinterpret_cast<float2*>(base + NA_PART_O);
  float* lse = reinterpret_cast<float*>(base + NA_PART_O + NA_PART_ML);

  qe::AttnParams p{};
  p.st = h->st;
  p.layer = layer;
  p.pend = m.pending;
  p.knew = m.pk;
  p.vnew = m.pv;
  p.cb = h->cost_b;
  p.cq = h->cost_q;
  p.pslots = NA_PSLOTS;
  p.q = static_cast<const uint16_t*>(q);
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.lse = lse;
  p.rope_blk = h->rope_blk;
  p.rope_off = h->rope_off;
  p.debug_expire = 0;
  const int grid = qe::attn_grid(h->n_sm, h->units, NA_PSLOTS);
  e = qe::launch_decode_attn(p, grid, h->stream);
  if (e != cudaSuccess) return na_fail(h, QE_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  m.pending = 0;
  m.pk = m.pv = nullptr;
  qe::CombineParams cp{};
  cp.st = h->st;
  cp.layer = layer;
  cp.pend = p.pend;
  cp.cb = p.cb;
  cp.cq = p.cq;
  cp.NW = grid * qe::attn_warps_per_cta();
  cp.pslots = NA_PSLOTS;
  cp.part_o = part_o;
  cp.part_ml = part_ml;
  cp.lse = lse;
  cp.out = out;
  cp.out_fp32 = h->cfg.out_fp32;
  e = qe::launch_attn_combine(cp, h->stream);
  if (e != cudaSuccess) return na_fail(h, QE_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
  h->launches += 2;
  return QE_OK;
}
