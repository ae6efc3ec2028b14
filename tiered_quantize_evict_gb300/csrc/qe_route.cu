// qe_route.cu -- append, routing (segmented top-K + tier diff + free-list bookkeeping) and
// window moves (first-demotion pack, ledger reuse, promotion) of the tiered KV cache.
//
// Sources: QEvict reading notes §4.4 eqs. (4)-(6) and Algorithm 1 (candidate pool, greedy
// TopK assignment, quantize once and reuse the ledger, promotion); HqeKV reading notes §2.3
// eq. (2) (z = min, s = (max - min) / (2^b - 1), nearest level); KV Cache technology
// evolution §5 (keys quantized per channel across tokens, values per token); H2O page §5.1
// (ties broken on the original position, in-place slot reuse, slot != position).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qe_kernels.cuh"

namespace qe {

// ------------------------------------------------------------------------------ append
// Every append kernel reads the layer's length from the device header and the last CTA to
// finish commits the new length, so the launch arguments never change from step to step.
__device__ __forceinline__ void commit_length(const State& st, int layer, int L_new) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    LayerDev* h = st.ldev + layer;
    if (atomicAdd(&h->done, 1u) == gridDim.x - 1) {
      h->L = L_new;
      h->done = 0;
      __threadfence();
    }
  }
}

// open window j of unit gu: pop a bf16 slot, Pinned, score 0, entry `nb` of the bf16 list
__device__ __forceinline__ int open_window(const State& st, long long gu, int j, int nb) {
  int top = st.bfree_top[gu];
  if (top <= 0 || nb >= st.capb) {
    atomicOr(st.err, ERR_FREELIST);
    return -1;
  }
  const int s = st.bfree[gu * st.capb + (--top)];
  st.bfree_top[gu] = top;
  st.bslot[gu * st.maxw + j] = s;
  st.tier[gu * st.maxw + j] = TIER_PINNED;
  st.score[gu * st.maxw + j] = 0.f;
  st.blist[gu * st.capb + nb] = make_int2(j, s);
  return s;
}

__device__ __forceinline__ void write_token(const State& st, long long gu, int slot, int row, int c, unsigned kk,
                                            uint16_t v0, uint16_t v1) {
  uint8_t* base = st.bslab + (gu * st.capb + slot) * (long long)st.geo.bslot_bytes();
  *reinterpret_cast<unsigned*>(base + bf16_k_off(st.geo, row, c)) = kk;
  *reinterpret_cast<uint16_t*>(base + bf16_v_off(st.geo, row, c)) = v0;
  *reinterpret_cast<uint16_t*>(base + bf16_v_off(st.geo, row, c + 1)) = v1;
}

// One decode token: APPEND1_UNITS units per CTA, one thread per channel pair.  The token that
// starts a window opens it (QEvict notes §2 Figure 1: every window starts in full precision).
// The length is not advanced here: the next decode step counts this token as pending and its
// combine launch commits the new length (see qe_decode_step), so the launch stays step-invariant.
constexpr int APPEND1_UNITS = 2;
__global__ void qe_append1_kernel(State st, int layer, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v) {
  __shared__ int s_slot[APPEND1_UNITS];
  const LayerDev hd = st.ldev[layer];
  const int L = hd.L, W = st.geo.W, D = st.geo.D;
  if (L + 1 > st.max_context) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(st.err, ERR_CAPACITY);
    return;
  }
  const int j = L / W;
  const int u0 = blockIdx.x * APPEND1_UNITS;
  if (threadIdx.x < APPEND1_UNITS && u0 + (int)threadIdx.x < st.units) {
    const long long gu = (long long)layer * st.units + u0 + threadIdx.x;
    int slot;
    if (L % W == 0) slot = open_window(st, gu, j, 1 + hd.n_full + (j - hd.routed_upto));
    else slot = st.bslot[gu * st.maxw + j];
    if (L < st.n_sink) slot = 0;
    s_slot[threadIdx.x] = slot;
  }
  __syncthreads();
  const int row = L < st.n_sink ? L : L - j * W;
  const int ul = threadIdx.x / (D / 2), c = 2 * (threadIdx.x % (D / 2));
  const int u = u0 + ul;
  if (ul >= APPEND1_UNITS || u >= st.units) return;
  const int slot = s_slot[ul];
  if (slot < 0 || slot >= st.capb || (slot == 0 && L >= st.n_sink)) {
    atomicOr(st.err, ERR_TABLE);
    return;
  }
  const long long gu = (long long)layer * st.units + u;
  const size_t src = (size_t)u * D + c;
  write_token(st, gu, slot, row, c, *reinterpret_cast<const unsigned*>(k + src), v[src], v[src + 1]);
}

// Advance the committed length of a layer by n (a single-token append that no decode step
// consumed).
__global__ void qe_commit_length_kernel(State st, int layer, int n) { st.ldev[layer].L += n; }

// Prefill part 1: open the windows [ceil(L/w), ceil((L+n)/w)) of every unit.  One thread per unit.
__global__ void qe_open_windows_kernel(State st, int layer, int n) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= st.units) return;
  const LayerDev hd = st.ldev[layer];
  if (hd.L + n > st.max_context) return;
  const int W = st.geo.W;
  const int w_old = (hd.L + W - 1) / W, w_new = (hd.L + n + W - 1) / W;
  const long long gu = (long long)layer * st.units + u;
  int nb = 1 + hd.n_full + (w_old - hd.routed_upto);
  for (int j = w_old; j < w_new; ++j, ++nb)
    if (open_window(st, gu, j, nb) < 0) break;
}

// Prefill part 2: copy n tokens (positions [L, L+n)) of K and V into their window slots in
// fragment order.  Thread per (unit, token, channel pair); sink positions go to the sink slot.
__global__ void qe_append_kernel(State st, int layer, int n, const uint16_t* __restrict__ k,
                                 const uint16_t* __restrict__ v) {
  const int D = st.geo.D, W = st.geo.W;
  const int pos0 = st.ldev[layer].L;
  if (pos0 + n > st.max_context) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(st.err, ERR_CAPACITY);
    commit_length(st, layer, pos0);
    return;
  }
  const long long total = (long long)st.units * n * (D / 2);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int cp = (int)(idx % (D / 2));
    const long long rest = idx / (D / 2);
    const int tk = (int)(rest % n);
    const int u = (int)(rest / n);
    const int pos = pos0 + tk;
    const int c = 2 * cp;
    const long long gu = (long long)layer * st.units + u;
    const size_t src = ((size_t)u * n + tk) * D + c;
    int slot, row;
    if (pos < st.n_sink) {
      slot = 0;
      row = pos;
    } else {
      const int j = pos / W;
      slot = st.bslot[gu * st.maxw + j];
      row = pos - j * W;
      if (slot <= 0 || slot >= st.capb) { atomicOr(st.err, ERR_TABLE); continue; }
    }
    write_token(st, gu, slot, row, c, *reinterpret_cast<const unsigned*>(k + src), v[src], v[src + 1]);
  }
  commit_length(st, layer, pos0 + n);
}

// ------------------------------------------------------------------------------ route
constexpr int ROUTE_THREADS = 256;
constexpr int ROUTE_MAX_CAND = 4096;

// One CTA per unit.  Shared memory: sort keys, per-kind change lists, the three free stacks.
__global__ void __launch_bounds__(ROUTE_THREADS) qe_route_kernel(const RouteParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const State& st = p.st;
  const int u = blockIdx.x;
  const long long gu = (long long)p.layer * st.units + u;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(sm);              // ROUTE_MAX_CAND
  int* ch_win = reinterpret_cast<int*>(keys + ROUTE_MAX_CAND);                       // ROUTE_MAX_CAND
  uint8_t* ch_new = reinterpret_cast<uint8_t*>(ch_win + ROUTE_MAX_CAND);             // ROUTE_MAX_CAND
  int* bstack = reinterpret_cast<int*>(ch_new + ROUTE_MAX_CAND);                     // capb
  int* qstack = bstack + st.capb;                                                    // capq
  int* sstack = qstack + st.capq;                                                    // caps
  __shared__ int s_n, s_nch, s_pos[2];
  __shared__ int s_moves_base;
  __shared__ int s_nmoves;

  const int tid = threadIdx.x;
  // this event's geometry and capacities, from the device-resident header (identical in every CTA)
  const LayerDev hd = st.ldev[p.layer];
  const int W = st.geo.W;
  const int L = hd.L;
  const int n_windows = (L + W - 1) / W;
  int aged_upto = (L - st.n_recent) >= 0 ? (L - st.n_recent) / W : 0;
  if (aged_upto < hd.routed_upto) aged_upto = hd.routed_upto;
  int kf, kq;
  capacities_at(st.cap, st.n_sink, st.n_recent, W, st.geo.D, L, kf, kq);
  const int ncand = hd.n_full + hd.n_quant + (aged_upto - hd.routed_upto);
  const int exp_nfull = kf < ncand ? kf : ncand;
  const int exp_nquant = kq < ncand - exp_nfull ? kq : ncand - exp_nfull;
  const bool fits = exp_nquant <= st.capq && exp_nfull + exp_nquant <= st.caps && ncand <= ROUTE_MAX_CAND;
  if (tid == 0) { s_n = 0; s_nch = 0; s_nmoves = 0; }
  __syncthreads();
  if (!fits) {   // the pools cannot hold this event's result: flag and leave the layer unchanged
    if (tid == 0 && u == 0) atomicOr(st.err, ERR_CAPACITY);
    return;
  }
  // 1. candidate pool, eq. (4): Full u Quantized u newly aged Pinned windows
  const uint8_t* tier = st.tier + gu * st.maxw;
  const float* score = st.score + gu * st.maxw;
  for (int j = tid; j < aged_upto; j += ROUTE_THREADS) {
    const int z = tier[j];
    const bool cand = (z == TIER_FULL) || (z == TIER_QUANT) || (z == TIER_PINNED && j >= hd.routed_upto);
    if (cand) {
      const int pos = atomicAdd(&s_n, 1);
      if (pos < ROUTE_MAX_CAND) {
        // ascending key order = score descending, then window ascending (scores are >= 0)
        const unsigned sb = __float_as_uint(score[j]);
        keys[pos] = ((unsigned long long)(0xFFFFFFFFu - sb) << 32) | (unsigned)j;
      }
    }
  }
  __syncthreads();
  if (tid == 0 && s_n > ROUTE_MAX_CAND) atomicOr(st.err, ERR_COUNT);
  const int n = s_n < ROUTE_MAX_CAND ? s_n : ROUTE_MAX_CAND;
  int npow = 1;
  while (npow < n) npow <<= 1;
  for (int i = n + tid; i < npow; i += ROUTE_THREADS) keys[i] = ~0ull;
  __syncthreads();
  // 2. bitonic sort of the keys
  for (int k = 2; k <= npow; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = tid; i < npow; i += ROUTE_THREADS) {
        const int ixj = i ^ jj;
        if (ixj > i) {
          const unsigned long long a = keys[i], b = keys[ixj];
          const bool up = (i & k) == 0;
          if ((a > b) == up) { keys[i] = b; keys[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
  // 3. eq. (5): rank -> tier; collect the windows whose tier changes
  for (int r = tid; r < n; r += ROUTE_THREADS) {
    const int j = (int)(keys[r] & 0xFFFFFFFFu);
    const int nt = r < kf ? TIER_FULL : (r < kf + kq ? TIER_QUANT : TIER_EVICTED);
    const int ot = tier[j];
    const int ot2 = ot == TIER_PINNED ? TIER_FULL : ot;   // Pinned -> Full moves no data
    if (nt != ot) {
      if (nt == ot2) {
        st.tier[gu * st.maxw + j] = (uint8_t)nt;
      } else {
        const int c = atomicAdd(&s_nch, 1);
        ch_win[c] = j;
        ch_new[c] = (uint8_t)nt;
      }
    }
  }
  // free stacks into shared memory
  const int btop = st.bfree_top[gu], qtop = st.qfree_top[gu], stop = st.sfree_top[gu];
  for (int i = tid; i < btop; i += ROUTE_THREADS) bstack[i] = st.bfree[gu * st.capb + i];
  for (int i = tid; i < qtop; i += ROUTE_THREADS) qstack[i] = st.qfree[gu * st.capq + i];
  for (int i = tid; i < stop; i += ROUTE_THREADS) sstack[i] = st.sfree[gu * st.caps + i];
  __syncthreads();
  // 4. bookkeeping, one thread, in an order that never hands out a slot whose data a move
  //    still has to read: 2-bit and store frees first (their contents are not needed),
  //    bf16 slots for promotions next, then demotions, then the bf16 frees.
  if (tid == 0) {
    const int nch = s_nch;
    int bt = btop, qt = qtop, stt = stop;
    unsigned err = 0;
    int nm = 0;
    int* bsl = st.bslot + gu * st.maxw;
    int* qsl = st.qslot + gu * st.maxw;
    int* sen = st.sent + gu * st.maxw;
    // (a) leaving the 2-bit pool: promotions and evictions of Quantized windows
    for (int c = 0; c < nch; ++c) {
      const int j = ch_win[c];
      if (tier[j] == TIER_QUANT) {
        const int s = qsl[j];
        if (s < 0 || qt >= st.capq) err |= ERR_FREELIST; else qstack[qt++] = s;
        qsl[j] = -1;
      }
    }
    // (b) evictions release their store / ledger entry
    for (int c = 0; c < nch; ++c) {
      const int j = ch_win[c];
      if (ch_new[c] == TIER_EVICTED && sen[j] >= 0) {
        if (stt >= st.caps) err |= ERR_FREELIST; else sstack[stt++] = sen[j];
        sen[j] = -1;
      }
    }
    // (c) promotions: a bf16 slot, filled from the exact host copy
    for (int c = 0; c < nch; ++c) {
      const int j = ch_win[c];
      if (ch_new[c] == TIER_FULL && tier[j] == TIER_QUANT) {
        if (bt <= 0 || sen[j] < 0) { err |= ERR_FREELIST; continue; }
        const int s = bstack[--bt];
        bsl[j] = s;
        keys[nm++] = ((unsigned long long)2 << 56) | ((unsigned long long)(unsigned)c << 24);
      }
    }
    // (d) demotions: a 2-bit slot; first demotion packs and takes a store entry, later ones reuse
    for (int c = 0; c < nch; ++c) {
      const int j = ch_win[c];
      if (ch_new[c] == TIER_QUANT) {
        if (qt <= 0) { err |= ERR_FREELIST; continue; }
        qsl[j] = qstack[--qt];
        if (sen[j] < 0) {
          if (stt <= 0) { err |= ERR_FREELIST; continue; }
          sen[j] = sstack[--stt];
          keys[nm++] = ((unsigned long long)0 << 56) | ((unsigned long long)(unsigned)c << 24);
        } else {
          keys[nm++] = ((unsigned long long)1 << 56) | ((unsigned long long)(unsigned)c << 24);
        }
      }
    }
    // (e) bf16 frees (after the moves above were decided; the move kernel reads them first)
    s_nmoves = nm;
    // write the move records (slot numbers captured before the frees below clear bslot)
    int base = 0;
    if (nm > 0) base = atomicAdd(p.n_moves, nm);
    s_moves_base = base;
    for (int k = 0; k < nm; ++k) {
      const int kind = (int)(keys[k] >> 56);
      const int c = (int)((keys[k] >> 24) & 0xFFFFFFFF);
      const int j = ch_win[c];
      Move mv;
      mv.kind = kind;
      mv.gu = (int)gu;
      mv.win = j;
      if (kind == 0) { mv.src = bsl[j]; mv.dst = qsl[j]; mv.sent = sen[j]; }
      else if (kind == 1) { mv.src = sen[j]; mv.dst = qsl[j]; mv.sent = sen[j]; }
      else { mv.src = sen[j]; mv.dst = bsl[j]; mv.sent = sen[j]; }
      if (base + k < p.max_moves) p.moves[base + k] = mv; else err |= ERR_MOVES;
    }
    for (int c = 0; c < nch; ++c) {
      const int j = ch_win[c];
      const int ot = tier[j];
      if ((ot == TIER_PINNED || ot == TIER_FULL) && ch_new[c] != TIER_FULL) {
        if (bsl[j] < 0 || bt >= st.capb) err |= ERR_FREELIST; else bstack[bt++] = bsl[j];
        bsl[j] = -1;
      }
    }
    // tier updates and statistics
    unsigned long long nfirst = 0, nreuse = 0, nprom = 0, nev = 0;
    for (int k = 0; k < nm; ++k) {
      const int kind = (int)(keys[k] >> 56);
      if (kind == 0) ++nfirst; else if (kind == 1) ++nreuse; else ++nprom;
    }
    for (int c = 0; c < nch; ++c) {
      st.tier[gu * st.maxw + ch_win[c]] = ch_new[c];
      if (ch_new[c] == TIER_EVICTED) ++nev;
    }
    unsigned long long* sp = st.stats + (size_t)p.layer * 5;
    if (u == 0) atomicAdd(sp + 0, 1ull);
    if (nfirst) atomicAdd(sp + 1, nfirst);
    if (nreuse) atomicAdd(sp + 2, nreuse);
    if (nprom) atomicAdd(sp + 3, nprom);
    if (nev) atomicAdd(sp + 4, nev);
    st.bfree_top[gu] = bt;
    st.qfree_top[gu] = qt;
    st.sfree_top[gu] = stt;
    s_pos[0] = bt;
    s_pos[1] = qt;
    if (err) atomicOr(st.err, err);
  }
  __syncthreads();
  {
    const int bt = s_pos[0], qt = s_pos[1], stt = st.sfree_top[gu];
    for (int i = tid; i < bt; i += ROUTE_THREADS) st.bfree[gu * st.capb + i] = bstack[i];
    for (int i = tid; i < qt; i += ROUTE_THREADS) st.qfree[gu * st.capq + i] = qstack[i];
    for (int i = tid; i < stt; i += ROUTE_THREADS) st.sfree[gu * st.caps + i] = sstack[i];
  }
  __syncthreads();
  // 5. rebuild the tile lists: bf16 = sink + Pinned/Full windows, 2-bit = Quantized windows,
  //    both in ascending window order (block-wide stream compaction)
  __shared__ int s_cnt[ROUTE_THREADS][2];
  const int per = (n_windows + ROUTE_THREADS - 1) / ROUTE_THREADS;
  const int j0 = tid * per, j1 = min(j0 + per, n_windows);
  int cb = 0, cq = 0;
  for (int j = j0; j < j1; ++j) {
    const int z = st.tier[gu * st.maxw + j];
    cb += (z == TIER_PINNED || z == TIER_FULL);
    cq += (z == TIER_QUANT);
  }
  s_cnt[tid][0] = cb;
  s_cnt[tid][1] = cq;
  __syncthreads();
  if (tid == 0) {
    int ab = 1, aq = 0;   // bf16 entry 0 is the sink
    for (int i = 0; i < ROUTE_THREADS; ++i) {
      const int b = s_cnt[i][0], q = s_cnt[i][1];
      s_cnt[i][0] = ab;
      s_cnt[i][1] = aq;
      ab += b;
      aq += q;
    }
    const int exp_b = 1 + exp_nfull + (n_windows - aged_upto);
    if (ab != exp_b || aq != exp_nquant) atomicOr(st.err, ERR_COUNT);
    st.blist[gu * st.capb] = make_int2(-1, 0);
  }
  __syncthreads();
  int ob = s_cnt[tid][0], oq = s_cnt[tid][1];
  for (int j = j0; j < j1; ++j) {
    const int z = st.tier[gu * st.maxw + j];
    if (z == TIER_PINNED || z == TIER_FULL) {
      if (ob < st.capb) st.blist[gu * st.capb + ob] = make_int2(j, st.bslot[gu * st.maxw + j]);
      ++ob;
    } else if (z == TIER_QUANT) {
      if (oq < st.capq) st.qlist[gu * st.capq + oq] = make_int2(j, st.qslot[gu * st.maxw + j]);
      ++oq;
    }
  }
  // 6. the last CTA commits the new counts to the layer header
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    LayerDev* h = st.ldev + p.layer;
    if (atomicAdd(&h->done, 1u) == gridDim.x - 1) {
      h->routed_upto = aged_upto;
      h->n_full = exp_nfull;
      h->n_quant = exp_nquant;
      h->kf = kf;
      h->kq = kq;
      h->done = 0;
      __threadfence();
    }
  }
}

// ------------------------------------------------------------------------------ moves
// Grid-stride over the move list; one CTA per move.
//  pack:      bf16 slot -> 2-bit slot (eq. (2), b = 2: keys per channel over the window's
//             valid tokens, values per token over head_dim), then the 2-bit slot and the
//             bf16 slot are copied to the host ledger / store entry (mapped pinned memory)
//  reuse:     host ledger entry -> 2-bit slot
//  promotion: host store entry -> bf16 slot
constexpr int MOVE_THREADS = 256;

__device__ __forceinline__ void copy16(uint8_t* dst, const uint8_t* src, int bytes, int tid, int nthr) {
  for (int o = tid * 16; o < bytes; o += nthr * 16)
    *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(src + o);
}

// eq. (2): code = clamp(rint((x - z) / s), 0, 3) with z = min, s = (max - min) / 3 in float32
__device__ __forceinline__ unsigned quant_code(float x, float z, float s) {
  if (s == 0.f) return 0u;
  float qv = rintf(__fdiv_rn(__fsub_rn(x, z), s));
  qv = fminf(fmaxf(qv, 0.f), 3.f);
  return (unsigned)qv;
}

__global__ void __launch_bounds__(MOVE_THREADS) qe_move_kernel(State st, const Move* __restrict__ moves,
                                                               const int* __restrict__ n_moves) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int n = *n_moves;
  const Geo g = st.geo;
  const int D = g.D, W = g.W;
  float* kf = reinterpret_cast<float*>(sm);          // [W][D]
  float* vf = kf + W * D;                            // [W][D]
  float* kz = vf + W * D;                            // [D]
  float* ks = kz + D;                                // [D]
  float* vz = ks + D;                                // [W]
  float* vs = vz + W;                                // [W]
  unsigned* words = reinterpret_cast<unsigned*>(vs + W);   // [2 * W * D / 16]
  const int tid = threadIdx.x;
  for (int mi = blockIdx.x; mi < n; mi += gridDim.x) {
    const Move mv = moves[mi];
    const long long gu = mv.gu;
    {
      const bool ok_gu = gu >= 0 && gu < (long long)st.units * st.n_layers;
      const bool ok = ok_gu && mv.win >= 0 && mv.win < st.maxw &&
                      (mv.kind == 2 ? (mv.src >= 0 && mv.src < st.caps && mv.dst > 0 && mv.dst < st.capb)
                                    : (mv.dst >= 0 && mv.dst < st.capq &&
                                       (mv.kind == 1 ? (mv.src >= 0 && mv.src < st.caps)
                                                     : (mv.src > 0 && mv.src < st.capb && mv.sent >= 0 &&
                                                        mv.sent < st.caps))));
      if (!ok) {
        if (tid == 0) atomicOr(st.err, ERR_MOVES);
        continue;
      }
    }
    if (mv.kind == 2) {
      const uint8_t* src = st.hstore + (gu * st.caps + mv.src) * (long long)g.bslot_bytes();
      uint8_t* dst = st.bslab + (gu * st.capb + mv.dst) * (long long)g.bslot_bytes();
      copy16(dst, src, g.bslot_bytes(), tid, MOVE_THREADS);
      continue;
    }
    if (mv.kind == 1) {
      const uint8_t* src = st.hledger + (gu * st.caps + mv.src) * (long long)g.qslot_bytes();
      uint8_t* dst = st.qslab + (gu * st.capq + mv.dst) * (long long)g.qslot_bytes();
      copy16(dst, src, g.qslot_bytes(), tid, MOVE_THREADS);
      continue;
    }
    // ---- pack
    const uint8_t* bs = st.bslab + (gu * st.capb + mv.src) * (long long)g.bslot_bytes();
    uint8_t* qs = st.qslab + (gu * st.capq + mv.dst) * (long long)g.qslot_bytes();
    const int lo = (mv.win == 0) ? st.n_sink : 0;
    for (int e = tid; e < W * D; e += MOVE_THREADS) {
      const int r = e / D, c = e - r * D;
      const uint16_t kb = *reinterpret_cast<const uint16_t*>(bs + bf16_k_off(g, r, c));
      const uint16_t vb = *reinterpret_cast<const uint16_t*>(bs + bf16_v_off(g, r, c));
      kf[e] = __uint_as_float((unsigned)kb << 16);
      vf[e] = __uint_as_float((unsigned)vb << 16);
    }
    __syncthreads();
    // key groups: one per channel over rows [lo, W); value groups: one per token over D
    for (int c = tid; c < D; c += MOVE_THREADS) {
      float mn = kf[lo * D + c], mx = mn;
      for (int r = lo + 1; r < W; ++r) {
        const float x = kf[r * D + c];
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
      kz[c] = mn;
      ks[c] = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
    }
    for (int r = tid; r < W; r += MOVE_THREADS) {
      float mn = vf[r * D], mx = mn;
      for (int c = 1; c < D; ++c) {
        const float x = vf[r * D + c];
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
      vz[r] = (r < lo) ? 0.f : mn;
      vs[r] = (r < lo) ? 0.f : __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
    }
    const int nwords = 2 * W * D / 16;
    for (int i = tid; i < nwords; i += MOVE_THREADS) words[i] = 0u;
    __syncthreads();
    // codes into their fragment words (word index = byte offset / 4)
    for (int e = tid; e < W * D; e += MOVE_THREADS) {
      const int r = e / D, c = e - r * D;
      const unsigned ck = (r < lo) ? 0u : quant_code(kf[e], kz[c], ks[c]);
      const unsigned cv = (r < lo) ? 0u : quant_code(vf[e], vz[r], vs[r]);
      const CodePos pk = kcode_pos(g, r, c);
      const CodePos pv = vcode_pos(g, r, c);
      atomicOr(&words[pk.byte >> 2], ck << pk.bit);
      atomicOr(&words[pv.byte >> 2], cv << pv.bit);
    }
    __syncthreads();
    for (int i = tid; i < nwords; i += MOVE_THREADS) reinterpret_cast<unsigned*>(qs)[i] = words[i];
    for (int c = tid; c < D; c += MOVE_THREADS) {
      reinterpret_cast<float*>(qs + g.off_kmin())[kparam_pos(c)] = kz[c];
      reinterpret_cast<float*>(qs + g.off_kscale())[kparam_pos(c)] = ks[c];
    }
    for (int r = tid; r < W; r += MOVE_THREADS) {
      reinterpret_cast<float*>(qs + g.off_vmin())[vparam_pos(g, r)] = vz[r];
      reinterpret_cast<float*>(qs + g.off_vscale())[vparam_pos(g, r)] = vs[r];
    }
    __syncthreads();
    // the ledger copy of the codes and the exact bf16 copy go to the mapped host store
    copy16(st.hledger + (gu * st.caps + mv.sent) * (long long)g.qslot_bytes(), qs, g.qslot_bytes(), tid,
           MOVE_THREADS);
    copy16(st.hstore + (gu * st.caps + mv.sent) * (long long)g.bslot_bytes(), bs, g.bslot_bytes(), tid,
           MOVE_THREADS);
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------ launchers
cudaError_t launch_append(const State& st, int layer, int n, const uint16_t* k, const uint16_t* v, int n_sm,
                          cudaStream_t s) {
  if (n == 1) {
    qe_append1_kernel<<<(st.units + APPEND1_UNITS - 1) / APPEND1_UNITS, APPEND1_UNITS * (st.geo.D / 2), 0, s>>>(
        st, layer, k, v);
    return cudaGetLastError();
  }
  qe_open_windows_kernel<<<(st.units + 127) / 128, 128, 0, s>>>(st, layer, n);
  const long long total = (long long)st.units * n * (st.geo.D / 2);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)n_sm * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  qe_append_kernel<<<(int)blocks, 256, 0, s>>>(st, layer, n, k, v);
  return cudaGetLastError();
}

cudaError_t launch_commit_length(const State& st, int layer, int n, cudaStream_t s) {
  qe_commit_length_kernel<<<1, 1, 0, s>>>(st, layer, n);
  return cudaGetLastError();
}

size_t route_smem_bytes(const State& st) {
  return (size_t)ROUTE_MAX_CAND * (8 + 4 + 1) + (size_t)(st.capb + st.capq + st.caps) * 4 + 16;
}

cudaError_t launch_route(const RouteParams& p, cudaStream_t s) {
  qe_route_kernel<<<p.st.units, ROUTE_THREADS, route_smem_bytes(p.st), s>>>(p);
  return cudaGetLastError();
}

size_t move_smem_bytes(const State& st) {
  const int W = st.geo.W, D = st.geo.D;
  return (size_t)(2 * W * D + 2 * D + 2 * W) * 4 + (size_t)(2 * W * D / 16) * 4;
}

cudaError_t launch_moves(const State& st, const Move* moves, const int* n_moves, int n_sm, cudaStream_t s) {
  qe_move_kernel<<<n_sm * 2, MOVE_THREADS, move_smem_bytes(st), s>>>(st, moves, n_moves);
  return cudaGetLastError();
}

// kernel attributes, set once (outside any stream capture)
cudaError_t prepare_route_kernels(const State& st) {
  cudaError_t e = cudaFuncSetAttribute(qe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)route_smem_bytes(st));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(qe_move_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)move_smem_bytes(st));
}

}  // namespace qe
