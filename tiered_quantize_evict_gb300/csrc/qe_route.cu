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

__device__ __forceinline__ void write_token(const State& st, long long gu, int slot, int row, int c, unsigned kk,
                                            uint16_t v0, uint16_t v1) {
  uint8_t* base = st.bslab + (gu * st.capb + slot) * (long long)st.geo.bslot_bytes();
  *reinterpret_cast<unsigned*>(base + bf16_k_off(st.geo, row, c)) = kk;
  *reinterpret_cast<uint16_t*>(base + bf16_v_off(st.geo, row, c)) = v0;
  *reinterpret_cast<uint16_t*>(base + bf16_v_off(st.geo, row, c + 1)) = v1;
}

// One single-token append that no decode step consumed (a decode step writes its pending
// token itself, inside the attention launch): APPEND1_UNITS units per CTA, one thread per
// channel pair.  The token that starts a window opens it (QEvict notes §2 Figure 1: every
// window starts in full precision).  The length is advanced by a separate commit launch.
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
                                 const uint16_t* __restrict__ v, int tok_major) {
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
    const size_t src = (tok_major ? (size_t)tk * st.units + u : (size_t)u * n + tk) * D + c;
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

// Block-wide exclusive prefix sum of one value per thread (ROUTE_THREADS threads, every thread
// calls it); returns this thread's prefix and sets *total.  s_w: ROUTE_THREADS / 32 + 1 ints of
// shared scratch, free again when the call returns.
__device__ int block_scan(int v, int* s_w, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_w[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < ROUTE_THREADS / 32 ? s_w[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < ROUTE_THREADS / 32) s_w[lane] = w;   // inclusive warp totals
  }
  __syncthreads();
  const int excl = (wid ? s_w[wid - 1] : 0) + x - v;
  *total = s_w[ROUTE_THREADS / 32 - 1];
  __syncthreads();
  return excl;
}

// Block-wide: write front[0, nf) and then the entries of rest[0, nr) whose slot is flagged free,
// in order, to dst (at most cap entries; more is a free-list error).  Returns the count on every
// thread.
__device__ int compact_free(const int* front, int nf, const int* rest, int nr, const uint8_t* flag, int* dst,
                            int cap, int* s_w, unsigned* err) {
  const int tid = threadIdx.x;
  const int per = (nr + ROUTE_THREADS - 1) / ROUTE_THREADS;
  const int i0 = tid * per, i1 = min(i0 + per, nr);
  auto keep = [&](int sl) { return sl >= 0 && sl < cap && flag[sl] != 0; };
  int cnt = 0;
  for (int i = i0; i < i1; ++i) cnt += keep(rest[i]);
  int kept;
  int o = nf + block_scan(cnt, s_w, &kept);
  const int acc = nf + kept;
  if (tid == 0 && acc > cap) atomicOr(err, ERR_FREELIST);
  for (int i = tid; i < nf && i < cap; i += ROUTE_THREADS) dst[i] = front[i];
  for (int i = i0; i < i1; ++i)
    if (keep(rest[i])) {
      if (o < cap) dst[o] = rest[i];
      ++o;
    }
  return acc < cap ? acc : cap;
}

// Candidate capacity of one unit's event: every candidate is a window below the current count,
// so the table's window capacity bounds it (and ROUTE_MAX_CAND bounds the shared memory).
__host__ __device__ inline int route_cand_cap(const State& st) {
  return st.maxw < ROUTE_MAX_CAND ? st.maxw : ROUTE_MAX_CAND;
}
// sort-key array length: the candidate capacity rounded up to a power of two
__host__ __device__ inline int route_key_cap(const State& st) {
  int k = 1;
  while (k < route_cand_cap(st)) k <<= 1;
  return k;
}

// One CTA per (unit, layer): blockIdx.x = unit, layer = p.layer + blockIdx.y, so one launch
// routes a run of layers.  Shared memory: sort keys, the changed windows' table entries, the
// free lists.
__global__ void __launch_bounds__(ROUTE_THREADS) qe_route_kernel(const RouteParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  const State& st = p.st;
  const int u = blockIdx.x;
  const int layer = p.layer + (int)blockIdx.y;
  const long long gu = (long long)layer * st.units + u;
  const int CC = route_cand_cap(st);
  // Changed windows carry a shared-memory copy of their table entries (old tier, bf16 slot,
  // 2-bit slot, store entry), so the serial bookkeeping below touches no global memory.
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(sm);              // route_key_cap
  int* ch_win = reinterpret_cast<int*>(keys + route_key_cap(st));                    // CC
  int* ch_b = ch_win + CC;                                                           // CC
  int* ch_q = ch_b + CC;                                                             // CC
  int* ch_s = ch_q + CC;                                                             // CC
  int* ch_bv = ch_s + CC;                  // previous bf16 slot still holding the window, or -1
  int* ch_qv = ch_bv + CC;                 // previous 2-bit slot still holding the window, or -1
  const int CC16 = (CC + 15) & ~15;
  uint8_t* ch_new = reinterpret_cast<uint8_t*>(ch_qv + CC);                          // CC16
  uint8_t* ch_old = ch_new + CC16;                                                   // CC16
  // free lists: the current entries (next to hand out first), then slots freed at the back;
  // slots freed at the front apart; a flag per slot says whether it is free
  int* bfa = reinterpret_cast<int*>(ch_old + CC16);                                  // 2 capb
  int* bfront = bfa + 2 * st.capb;                                                   // capb
  int* qfa = bfront + st.capb;                                                       // 2 capq
  int* qfront = qfa + 2 * st.capq;                                                   // capq
  int* sstack = qfront + st.capq;                                                    // caps
  // per 2-bit slot: the change-list index of the window promoted in this event whose codes the
  // slot still holds, else -1 (its store entry's flags then live in ch_s, not in the table)
  int* qch = sstack + st.caps;                                                       // capq
  uint8_t* bflag = reinterpret_cast<uint8_t*>(qch + st.capq);                        // capb
  uint8_t* qflag = bflag + st.capb;                                                  // capq
  __shared__ int s_n, s_nch, s_pos[8];
  __shared__ int s_diag[9];   // full old/new/both, kept old/new/both, promotions, demotions, evictions
  __shared__ float s_cut[4];  // scores at the two cuts (read before the keys are reused)
  __shared__ int s_w[ROUTE_THREADS / 32 + 1];

  const int tid = threadIdx.x;
  // this event's geometry and capacities, from the device-resident header (identical in every CTA)
  const LayerDev hd = st.ldev[layer];
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
  const bool fits = exp_nquant <= st.capq && exp_nfull + exp_nquant <= st.caps && ncand <= CC;
  if (tid == 0) { s_n = 0; s_nch = 0; }
  if (tid < 9) s_diag[tid] = 0;
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
      if (pos < CC) {
        // ascending key order = score descending, then window ascending (scores are >= 0)
        const unsigned sb = __float_as_uint(score[j]);
        keys[pos] = ((unsigned long long)(0xFFFFFFFFu - sb) << 32) | (unsigned)j;
      }
    }
  }
  __syncthreads();
  if (tid == 0 && s_n > CC) atomicOr(st.err, ERR_COUNT);
  const int n = s_n < CC ? s_n : CC;
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
  if (tid < 4) {
    const int r = tid < 2 ? kf - 1 + tid : kf + kq - 1 + (tid - 2);
    s_cut[tid] = (r >= 0 && r < n) ? __uint_as_float(0xFFFFFFFFu - (unsigned)(keys[r] >> 32)) : -1.f;
  }
  // 3. eq. (5): rank -> tier; collect the windows whose tier changes
  int* bsl = st.bslot + gu * st.maxw;
  int* qsl = st.qslot + gu * st.maxw;
  int* sen = st.sent + gu * st.maxw;
  int dg[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};   // this thread's share of the event record
  auto new_tier = [&](int r) { return r < kf ? TIER_FULL : (r < kf + kq ? TIER_QUANT : TIER_EVICTED); };
  int myc = 0;
  for (int r = tid; r < n; r += ROUTE_THREADS) {
    const int j = (int)(keys[r] & 0xFFFFFFFFu);
    const int nt = new_tier(r);
    const int ot = tier[j];
    const bool fo = ot == TIER_FULL, fn = nt == TIER_FULL;
    const bool ko = fo || ot == TIER_QUANT, kn = fn || nt == TIER_QUANT;
    dg[0] += fo; dg[1] += fn; dg[2] += fo && fn;
    dg[3] += ko; dg[4] += kn; dg[5] += ko && kn;
    dg[6] += ot == TIER_QUANT && fn;
    dg[7] += fo && nt == TIER_QUANT;
    dg[8] += nt == TIER_EVICTED;
    myc += nt != ot;
  }
  // the change list in a fixed order (thread, then rank), so slot hand-out is reproducible
  int nch_total;
  int c = block_scan(myc, s_w, &nch_total);
  if (tid == 0) s_nch = nch_total;
  for (int r = tid; r < n; r += ROUTE_THREADS) {
    const int j = (int)(keys[r] & 0xFFFFFFFFu);
    const int nt = new_tier(r);
    const int ot = tier[j];
    if (nt == ot) continue;
    ch_win[c] = j;
    ch_new[c] = (uint8_t)nt;
    ch_old[c] = (uint8_t)ot;
    ch_b[c] = bsl[j];
    ch_q[c] = qsl[j];
    ch_s[c] = sen[j];
    // the slot the window last held, if its contents are still the window's (a window leaving
    // Full for eviction also needs its 2-bit slot, whose codes must then never be saved)
    int bv = -1, qv = -1;
    if (nt == TIER_FULL && ot == TIER_QUANT) {
      const int sb = st.bprev[gu * st.maxw + j];
      if (sb > 0 && sb < st.capb && st.bvictim[gu * st.capb + sb] == j) bv = sb;
    }
    if (nt == TIER_QUANT || (nt == TIER_EVICTED && ot == TIER_FULL)) {
      const int sq = st.qprev[gu * st.maxw + j];
      if (sq >= 0 && sq < st.capq && st.qvictim[gu * st.capq + sq] == j) qv = sq;
    }
    ch_bv[c] = bv;
    ch_qv[c] = qv;
    ++c;
  }
  for (int i = 0; i < 9; ++i)
    if (dg[i]) atomicAdd(&s_diag[i], dg[i]);
  // free lists into shared memory
  const int bhead = st.bfree_head[gu], btop = st.bfree_top[gu], qtop = st.qfree_top[gu], stop = st.sfree_top[gu];
  const int nbf = btop > bhead ? btop - bhead : 0;
  for (int i = tid; i < st.capb; i += ROUTE_THREADS) bflag[i] = 0;
  for (int i = tid; i < st.capq; i += ROUTE_THREADS) {
    qflag[i] = 0;
    qch[i] = -1;
  }
  __syncthreads();
  for (int i = tid; i < nbf; i += ROUTE_THREADS) {
    const int sl = st.bfree[gu * st.capb + bhead + i];
    bfa[i] = sl;
    if (sl >= 0 && sl < st.capb) bflag[sl] = 1;
  }
  for (int i = tid; i < qtop; i += ROUTE_THREADS) {
    const int sl = st.qfree[gu * st.capq + i];
    qfa[i] = sl;
    if (sl >= 0 && sl < st.capq) qflag[sl] = 1;
  }
  for (int i = tid; i < stop; i += ROUTE_THREADS) sstack[i] = st.sfree[gu * st.caps + i];
  __syncthreads();
  const int nch = s_nch;
  // 4. bookkeeping, one thread, on the shared copies, in an order that never hands out a slot
  //    whose data a move still has to read: slots of evicted windows and 2-bit slots first
  //    (their contents are not needed), then promotions (taking back their previous slot when
  //    it still holds them), then demotions, then the bf16 slots of demoted windows (at the back).
  if (tid == 0) {
    int bh = 0, bn = nbf, bf_n = 0, bf_i = 0;   // bf16: pop cursor, end, front count, front cursor
    int qh = 0, qn = qtop, qf_n = 0, qf_i = 0;
    int stt = stop;
    unsigned err = 0;
    int nm = 0;
    // every list entry is a slot in range (only in-range slots are ever added)
    auto pop_b = [&]() -> int {
      if (bf_i < bf_n) { const int sl = bfront[bf_i++]; bflag[sl] = 0; return sl; }
      while (bh < bn && !(bfa[bh] > 0 && bfa[bh] < st.capb && bflag[bfa[bh]])) ++bh;
      if (bh >= bn) return -1;
      const int sl = bfa[bh++];
      bflag[sl] = 0;
      return sl;
    };
    auto pop_q = [&]() -> int {
      if (qf_i < qf_n) { const int sl = qfront[qf_i++]; qflag[sl] = 0; return sl; }
      while (qh < qn && !(qfa[qh] >= 0 && qfa[qh] < st.capq && qflag[qfa[qh]])) ++qh;
      if (qh >= qn) return -1;
      const int sl = qfa[qh++];
      qflag[sl] = 0;
      return sl;
    };
    unsigned long long nfirst = 0, nreuse = 0, nprom = 0, nev = 0, brec = 0, qrec = 0, nwb = 0;
    // (a) leaving the 2-bit pool: a promoted window's slot keeps its codes (back), an evicted
    //     window's slot goes to the front
    for (int c = 0; c < nch; ++c) {
      if (ch_old[c] != TIER_QUANT) continue;
      const int sl = ch_q[c];
      if (sl < 0 || sl >= st.capq) { err |= ERR_FREELIST; ch_q[c] = -1; continue; }
      if (ch_new[c] == TIER_EVICTED) {
        qfront[qf_n++] = sl;
        st.qvictim[gu * st.capq + sl] = -1;
      } else {
        qfa[qn++] = sl;
        qch[sl] = c;
        st.qprev[gu * st.maxw + ch_win[c]] = sl;
      }
      qflag[sl] = 1;
      ch_q[c] = -1;
    }
    // (b) evictions release their store / ledger entry and their bf16 slot (front)
    for (int c = 0; c < nch; ++c) {
      if (ch_new[c] != TIER_EVICTED) continue;
      ++nev;
      if (ch_s[c] >= 0) {
        if (stt >= st.caps) err |= ERR_FREELIST; else sstack[stt++] = ch_s[c] & ~SENT_FLAGS;
        ch_s[c] = -1;
      }
      // a Full window's codes left in a free 2-bit slot die with it: never saved to its entry
      if (ch_old[c] == TIER_FULL && ch_qv[c] >= 0) st.qvictim[gu * st.capq + ch_qv[c]] = -1;
      if (ch_old[c] == TIER_PINNED || ch_old[c] == TIER_FULL) {
        const int sl = ch_b[c];
        if (sl <= 0 || sl >= st.capb) err |= ERR_FREELIST;
        else {
          bfront[bf_n++] = sl;
          bflag[sl] = 1;
          st.bvictim[gu * st.capb + sl] = -1;
        }
        ch_b[c] = -1;
      }
    }
    // (c) promotions: the previous slot if it still holds the window, else a free slot filled
    //     from the exact host copy; Pinned windows kept Full get a store entry and their exact
    //     copy is written now
    for (int c = 0; c < nch; ++c) {
      if (ch_new[c] != TIER_FULL || ch_old[c] != TIER_QUANT) continue;
      const int sv = ch_bv[c];
      if (sv > 0 && bflag[sv]) {
        bflag[sv] = 0;
        ch_b[c] = sv;
        ch_bv[c] = -2;   // taken back: no move
        ++brec;
      }
    }
    for (int c = 0; c < nch; ++c) {
      if (ch_new[c] != TIER_FULL) continue;
      if (ch_old[c] == TIER_QUANT) {
        ++nprom;
        if (ch_bv[c] == -2) continue;
        if (ch_s[c] < 0) { err |= ERR_FREELIST; continue; }
        const int sl = pop_b();
        if (sl <= 0) { err |= ERR_FREELIST; continue; }
        ch_b[c] = sl;
        st.bvictim[gu * st.capb + sl] = ch_win[c];
        keys[nm++] = ((unsigned long long)MOVE_PROMOTE << 56) | ((unsigned long long)(unsigned)c << 24);
      } else if (ch_s[c] < 0) {
        if (stt <= 0) { err |= ERR_FREELIST; continue; }
        ch_s[c] = sstack[--stt];
        keys[nm++] = ((unsigned long long)MOVE_COPY << 56) | ((unsigned long long)(unsigned)c << 24);
      }
    }
    // (d) demotions: the previous 2-bit slot if it still holds the window's codes, else a free
    //     slot: the first demotion packs (and, from Pinned, takes a store entry for the exact
    //     copy), later ones copy the codes back from the host ledger
    for (int c = 0; c < nch; ++c) {
      if (ch_new[c] != TIER_QUANT) continue;
      const int qv = ch_qv[c];
      if (qv >= 0 && ch_s[c] >= 0 && (ch_s[c] & SENT_PACKED) && qflag[qv]) {
        qflag[qv] = 0;
        ch_q[c] = qv;
        ch_qv[c] = -2;
        ++qrec;
      }
    }
    for (int c = 0; c < nch; ++c) {
      if (ch_new[c] != TIER_QUANT) continue;
      if (ch_qv[c] == -2) { ++nreuse; continue; }
      const int sl = pop_q();
      if (sl < 0) { err |= ERR_FREELIST; continue; }
      // The slot may still hold the codes of a kept window (Full since an earlier event) whose
      // ledger was never written to the host: the move saves them to that window's entry
      // before it overwrites the slot.
      int wb = -1;
      {
        const int jo = st.qvictim[gu * st.capq + sl];
        if (jo >= 0 && jo < st.maxw && jo != ch_win[c]) {
          const int co = qch[sl];
          const int so = co >= 0 ? ch_s[co] : sen[jo];
          if (so >= 0 && (so & SENT_PACKED) && !(so & SENT_LEDGER)) {
            wb = so & ~SENT_FLAGS;
            if (co >= 0) ch_s[co] = so | SENT_LEDGER; else sen[jo] = so | SENT_LEDGER;
            ++nwb;
          }
        }
      }
      ch_qv[c] = wb;
      ch_q[c] = sl;
      st.qvictim[gu * st.capq + sl] = ch_win[c];
      int kind;
      if (ch_s[c] < 0) {
        if (stt <= 0) { err |= ERR_FREELIST; continue; }
        ch_s[c] = sstack[--stt];
        kind = MOVE_PACK_COPY;
      } else if (ch_s[c] & SENT_PACKED) {
        kind = MOVE_REUSE;   // the codes' only copy is the host ledger by now
        if (!(ch_s[c] & SENT_LEDGER)) err |= ERR_FREELIST;
      } else {
        kind = MOVE_PACK;
      }
      if (kind == MOVE_REUSE) ++nreuse; else ++nfirst;
      ch_s[c] |= SENT_PACKED;
      keys[nm++] = ((unsigned long long)kind << 56) | ((unsigned long long)(unsigned)c << 24);
    }
    // move records (slot numbers captured before the bf16 frees below clear them)
    int base = 0;
    if (nm > 0) base = atomicAdd(p.n_moves, nm);
    for (int k = 0; k < nm; ++k) {
      const int kind = (int)(keys[k] >> 56);
      const int c = (int)((keys[k] >> 24) & 0xFFFFFFFF);
      const int ent = ch_s[c] & ~SENT_FLAGS;
      Move mv;
      mv.kind = kind;
      mv.gu = (int)gu;
      mv.win = ch_win[c];
      mv.sent = ent;
      mv.wb = (kind == MOVE_PACK_COPY || kind == MOVE_PACK || kind == MOVE_REUSE) ? ch_qv[c] : -1;
      if (kind == MOVE_PACK_COPY || kind == MOVE_PACK) { mv.src = ch_b[c]; mv.dst = ch_q[c]; }
      else if (kind == MOVE_REUSE) { mv.src = ent; mv.dst = ch_q[c]; }
      else if (kind == MOVE_PROMOTE) { mv.src = ent; mv.dst = ch_b[c]; }
      else { mv.src = ch_b[c]; mv.dst = ent; }
      if (base + k < p.max_moves) p.moves[base + k] = mv; else err |= ERR_MOVES;
    }
    // (e) bf16 slots of demoted windows go to the back and keep the window's data (the move
    //     kernel reads them first)
    for (int c = 0; c < nch; ++c) {
      if (ch_new[c] != TIER_QUANT || (ch_old[c] != TIER_PINNED && ch_old[c] != TIER_FULL)) continue;
      const int sl = ch_b[c];
      if (sl <= 0 || sl >= st.capb) err |= ERR_FREELIST;
      else {
        bfa[bn++] = sl;
        bflag[sl] = 1;
        st.bprev[gu * st.maxw + ch_win[c]] = sl;
      }
      ch_b[c] = -1;
    }
    unsigned long long* sp = st.stats + (size_t)layer * N_STATS;
    if (u == 0) atomicAdd(sp + 0, 1ull);
    if (nfirst) atomicAdd(sp + 1, nfirst);
    if (nreuse) atomicAdd(sp + 2, nreuse);
    if (nprom) atomicAdd(sp + 3, nprom);
    if (nev) atomicAdd(sp + 4, nev);
    if (brec) atomicAdd(sp + 5, brec);
    if (qrec) atomicAdd(sp + 6, qrec);
    if (nwb) atomicAdd(sp + 7, nwb);
    st.sfree_top[gu] = stt;
    s_pos[0] = bh;
    s_pos[1] = bn;
    s_pos[2] = bf_i;
    s_pos[3] = bf_n;
    s_pos[4] = qh;
    s_pos[5] = qn;
    s_pos[6] = qf_i;
    s_pos[7] = qf_n;
    if (err) atomicOr(st.err, err);
  }
  __syncthreads();
  {
    // table entries and tiers of the changed windows, and the store stack, back to global memory
    for (int c = tid; c < nch; c += ROUTE_THREADS) {
      const int j = ch_win[c];
      bsl[j] = ch_b[c];
      qsl[j] = ch_q[c];
      sen[j] = ch_s[c];
      st.tier[gu * st.maxw + j] = ch_new[c];
    }
    for (int i = tid; i < st.sfree_top[gu]; i += ROUTE_THREADS) st.sfree[gu * st.caps + i] = sstack[i];
  }
  // the free lists, compacted: front entries not handed out, then the free entries in order
  {
    const int bh = s_pos[0], bn = s_pos[1], bf_i = s_pos[2], bf_n = s_pos[3];
    const int nb = compact_free(bfront + bf_i, bf_n - bf_i, bfa + bh, bn - bh, bflag, st.bfree + gu * st.capb,
                                st.capb, s_w, st.err);
    const int qh = s_pos[4], qn = s_pos[5], qf_i = s_pos[6], qf_n = s_pos[7];
    const int nq2 = compact_free(qfront + qf_i, qf_n - qf_i, qfa + qh, qn - qh, qflag, st.qfree + gu * st.capq,
                                 st.capq, s_w, st.err);
    if (tid == 0) {
      st.bfree_head[gu] = 0;
      st.bfree_top[gu] = nb;
      st.qfree_top[gu] = nq2;
    }
  }
  __syncthreads();
  // the event's record of this unit
  if (tid == 0 && p.diag) {
    RouteDiag d;
    d.kf = kf;
    d.kq = kq;
    d.full_old = s_diag[0]; d.full_new = s_diag[1]; d.full_both = s_diag[2];
    d.kept_old = s_diag[3]; d.kept_new = s_diag[4]; d.kept_both = s_diag[5];
    d.promotions = s_diag[6]; d.demotions = s_diag[7]; d.evictions = s_diag[8];
    d.full_cut_kept = s_cut[0];
    d.full_cut_next = s_cut[1];
    d.kept_cut_kept = s_cut[2];
    d.kept_cut_next = s_cut[3];
    p.diag[(size_t)layer * st.units + u] = d;
  }
  // 5. rebuild the tile lists: bf16 = sink + Pinned/Full windows, 2-bit = Quantized windows,
  //    both in ascending window order (block-wide stream compaction)
  const int per = (n_windows + ROUTE_THREADS - 1) / ROUTE_THREADS;
  const int j0 = tid * per, j1 = min(j0 + per, n_windows);
  int cb = 0, cq = 0;
  for (int j = j0; j < j1; ++j) {
    const int z = st.tier[gu * st.maxw + j];
    cb += (z == TIER_PINNED || z == TIER_FULL);
    cq += (z == TIER_QUANT);
  }
  int tb, tq;
  const int ob0 = 1 + block_scan(cb, s_w, &tb);   // bf16 entry 0 is the sink
  const int oq0 = block_scan(cq, s_w, &tq);
  if (tid == 0) {
    const int exp_b = 1 + exp_nfull + (n_windows - aged_upto);
    if (1 + tb != exp_b || tq != exp_nquant) atomicOr(st.err, ERR_COUNT);
    st.blist[gu * st.capb] = make_int2(-1, 0);
  }
  int ob = ob0, oq = oq0;
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
    LayerDev* h = st.ldev + layer;
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
// Grid-stride over the move list; one CTA per move.  The host ledger and store are mapped
// pinned memory, read and written directly over the host link.
//  pack:      bf16 slot -> 2-bit slot (eq. (2), b = 2: keys per channel over the window's
//             valid tokens, values per token over head_dim), and the codes to the host ledger;
//             from Pinned also the exact bf16 copy to the store entry
//  copy:      bf16 slot -> host store entry (a Pinned window kept Full)
//  reuse:     host ledger entry -> 2-bit slot
//  promotion: host store entry -> bf16 slot
constexpr int MOVE_THREADS = 256;
constexpr int MOVE_CTAS_PER_SM = 3;

// Copy `bytes` (a multiple of 16) with every thread's 16-byte loads issued before its stores,
// so a CTA keeps up to 4 x 4 KB in flight (the host side of a move is latency-bound).
__device__ __forceinline__ void copy16(uint8_t* dst, const uint8_t* src, int bytes, int tid) {
  constexpr int STEP = MOVE_THREADS * 16;
  for (int o0 = 0; o0 < bytes; o0 += 4 * STEP) {
    uint4 x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int o = o0 + i * STEP + tid * 16;
      if (o < bytes) x[i] = *reinterpret_cast<const uint4*>(src + o);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int o = o0 + i * STEP + tid * 16;
      if (o < bytes) *reinterpret_cast<uint4*>(dst + o) = x[i];
    }
  }
}

// eq. (2): code = clamp(rint((x - z) / s), 0, 3) with z = min, s = (max - min) / 3 in float32,
// the quotient rounded as IEEE float32 division rounds it.  For q = fl(d / s) >= 0 that code is
// [q > 1/2] + [q >= 3/2] + [q > 5/2] (rint ties to even: 1/2 -> 0, 3/2 -> 2, 5/2 -> 2), and as
// fl(d / s) never decreases with d, each term is [d >= T] for the smallest float T that passes
// it.  A group finds its three T once (a few correctly rounded divisions next to t s); each
// element then needs one subtraction and three compares.

// the code of one element by the division itself (groups whose thresholds are not searched)
__device__ __forceinline__ unsigned quant_code_div(float x, float z, float s) {
  if (s == 0.f) return 0u;
  float qv = rintf(__fdiv_rn(__fsub_rn(x, z), s));
  qv = fminf(fmaxf(qv, 0.f), 3.f);
  return (unsigned)qv;
}

// smallest non-negative float d with fl(d / s) > t (strict) or >= t; ok = false if it is not
// within 8 steps of fl(t s)
__device__ __forceinline__ float quant_threshold(float s, float t, bool strict, bool& ok) {
  auto pass = [&](float d) {
    const float q = __fdiv_rn(d, s);
    return strict ? q > t : q >= t;
  };
  float T = __fmul_rn(t, s);
  int i = 0;
  while (!pass(T) && i < 8) {
    T = __uint_as_float(__float_as_uint(T) + 1u);
    ++i;
  }
  if (i == 8) ok = false;
  i = 0;
  while (T > 0.f && i < 8 && pass(__uint_as_float(__float_as_uint(T) - 1u))) {
    T = __uint_as_float(__float_as_uint(T) - 1u);
    ++i;
  }
  if (i == 8) ok = false;
  return T;
}

// The thresholds of a group with scale s, found by its TPG threads (part k finds T_k, T_k+TPG,
// ...): {T_1/2, T_3/2, T_5/2}, or T_1/2 = -1 where the group's elements take the division (a
// scale outside [1e-30, 1e30], or a search that did not settle).  s = 0: every code is 0.
template <int TPG>
__device__ __forceinline__ void group_thresholds(float s, int part, float (&T)[3]) {
  const bool ranged = s >= 1e-30f && s <= 1e30f;
  bool ok = true;
  float mine[2] = {INFINITY, INFINITY};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int k = part + j * TPG;
    if (ranged && k < 3) mine[j] = quant_threshold(s, 0.5f + k, k != 1, ok);
  }
  unsigned okv = ok ? 1u : 0u;
#pragma unroll
  for (int o = 1; o < TPG; o <<= 1) okv &= __shfl_xor_sync(0xffffffffu, okv, o);
  const int base = (threadIdx.x & 31) & ~(TPG - 1);
#pragma unroll
  for (int k = 0; k < 3; ++k) T[k] = __shfl_sync(0xffffffffu, mine[k / TPG], base + k % TPG);
  if (s == 0.f) T[0] = T[1] = T[2] = INFINITY;
  else if (!ranged || !okv) T[0] = -1.f;
}

__device__ __forceinline__ unsigned quant_code(float x, const float4& p, float s) {
  if (p.y < 0.f) return quant_code_div(x, p.x, s);
  const float d = __fsub_rn(x, p.x);
  return (unsigned)(d >= p.y) + (unsigned)(d >= p.z) + (unsigned)(d >= p.w);
}

__device__ __forceinline__ float bf16_at(const uint8_t* raw, int off) {
  return __uint_as_float((unsigned)*reinterpret_cast<const uint16_t*>(raw + off) << 16);
}

// every index of a move record in range for its kind
__device__ __forceinline__ bool move_ok(const State& st, const Move& mv) {
  const bool ok_gu = mv.gu >= 0 && (long long)mv.gu < (long long)st.units * st.n_layers;
  const bool src_store = mv.src >= 0 && mv.src < st.caps, src_bf16 = mv.src > 0 && mv.src < st.capb;
  const bool dst_q = mv.dst >= 0 && mv.dst < st.capq, sent_ok = mv.sent >= 0 && mv.sent < st.caps;
  const bool ok = ok_gu && mv.win >= 0 && mv.win < st.maxw && mv.wb >= -1 && mv.wb < st.caps;
  switch (mv.kind) {
    case MOVE_PROMOTE: return ok && src_store && mv.dst > 0 && mv.dst < st.capb;
    case MOVE_REUSE: return ok && src_store && dst_q;
    case MOVE_PACK_COPY:
    case MOVE_PACK: return ok && src_bf16 && dst_q && sent_ok;
    case MOVE_COPY: return ok && src_bf16 && mv.dst >= 0 && mv.dst < st.caps;
    default: return false;
  }
}

// Each CTA takes every gridDim.x-th move.  A pack's bf16 source slot is fetched into one of two
// shared-memory buffers by asynchronous copies issued one move ahead, so it lands while the
// CTA works on the move before.
// Range record (qrange_word) of the codes 2-bit slot `slot` of unit gu now holds, from its key
// scales ks[D] and value scales vs[W] (any order); executed by one warp.
__device__ __forceinline__ void write_qrange(const State& st, long long gu, int slot, const float* ks, const float* vs,
                                             int D, int W, int lane) {
  unsigned kmax = 0u, vmax = 0u, vmin = 0xFFFFFFFFu;
  for (int c = lane; c < D; c += 32) kmax = max(kmax, __float_as_uint(ks[c]));
  for (int r = lane; r < W; r += 32) {
    const unsigned b = __float_as_uint(vs[r]);
    vmax = max(vmax, b);
    if (b) vmin = min(vmin, b);
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  vmax = __reduce_max_sync(0xffffffffu, vmax);
  vmin = __reduce_min_sync(0xffffffffu, vmin);
  if (lane == 0) st.qrange[gu * st.capq + slot] = qrange_word(kmax, vmax, vmin);
}

template <int D, int W>
__global__ void __launch_bounds__(MOVE_THREADS, MOVE_CTAS_PER_SM) qe_move_kernel(State st, const Move* __restrict__ moves,
                                                                                const int* __restrict__ n_moves) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int n = *n_moves;
  const Geo g{D, W};
  constexpr int BSLOT = 4 * W * D, QSLOT = 2 * (W * D / 4) + 8 * D + 8 * W;
  uint8_t* rawbuf[2] = {sm, sm + BSLOT};                               // bf16 slots [4 W D]
  float4* kp = reinterpret_cast<float4*>(sm + 2 * BSLOT);              // [D] {min, T_1/2, T_3/2, T_5/2}
  float4* vp = kp + D;                                                 // [W]
  float* kz = reinterpret_cast<float*>(vp + W);                        // [D]
  float* ks = kz + D;                                                  // [D]
  float* vz = ks + D;                                                  // [W]
  float* vs = vz + W;                                                  // [W]
  uint8_t* qimg = reinterpret_cast<uint8_t*>(vs + W);                  // the packed 2-bit slot
  const int tid = threadIdx.x;
  auto is_pack = [](int kind) { return kind == MOVE_PACK || kind == MOVE_PACK_COPY; };
  // one commit group per move (empty unless the move is a valid pack)
  auto prefetch = [&](int m, int b) {
    if (m < n) {
      const Move mv = moves[m];
      if (is_pack(mv.kind) && move_ok(st, mv)) {
        const uint8_t* src = st.bslab + ((long long)mv.gu * st.capb + mv.src) * (long long)BSLOT;
        for (int o = tid * 16; o < BSLOT; o += MOVE_THREADS * 16) cp_async16(rawbuf[b] + o, src + o);
      }
    }
    cp_async_commit();
  };
  int cur = 0;
  prefetch(blockIdx.x, 0);
  for (int mi = blockIdx.x; mi < n; mi += gridDim.x, cur ^= 1) {
    const Move mv = moves[mi];
    // The other buffer's last reader was the move two back, which ended with a barrier.
    prefetch(mi + gridDim.x, cur ^ 1);
    const long long gu = mv.gu;
    if (!move_ok(st, mv)) {
      if (tid == 0) atomicOr(st.err, ERR_MOVES);
      continue;
    }
    if (mv.kind == MOVE_PROMOTE) {
      const uint8_t* src = st.hstore + (gu * st.caps + mv.src) * (long long)BSLOT;
      uint8_t* dst = st.bslab + (gu * st.capb + mv.dst) * (long long)BSLOT;
      copy16(dst, src, BSLOT, tid);
      continue;
    }
    if (mv.kind == MOVE_COPY) {
      const uint8_t* src = st.bslab + (gu * st.capb + mv.src) * (long long)BSLOT;
      uint8_t* dst = st.hstore + (gu * st.caps + mv.dst) * (long long)BSLOT;
      copy16(dst, src, BSLOT, tid);
      continue;
    }
    if (mv.wb >= 0) {   // save the codes the 2-bit slot still holds for a kept window first
      const uint8_t* src = st.qslab + (gu * st.capq + mv.dst) * (long long)QSLOT;
      uint8_t* dst = st.hledger + (gu * st.caps + mv.wb) * (long long)QSLOT;
      copy16(dst, src, QSLOT, tid);
      __syncthreads();
    }
    if (mv.kind == MOVE_REUSE) {
      const uint8_t* src = st.hledger + (gu * st.caps + mv.src) * (long long)QSLOT;
      uint8_t* dst = st.qslab + (gu * st.capq + mv.dst) * (long long)QSLOT;
      copy16(dst, src, QSLOT, tid);
      __syncthreads();
      // the slot's range record, from the parameters it now holds
      if (tid < 32)
        write_qrange(st, gu, mv.dst, reinterpret_cast<const float*>(dst + g.off_kscale()),
                     reinterpret_cast<const float*>(dst + g.off_vscale()), D, W, tid);
      __syncthreads();
      continue;
    }
    // ---- pack: the bf16 slot (fetched one move ahead), and its exact copy into the host store
    const uint8_t* raw = rawbuf[cur];
    uint8_t* qs = st.qslab + (gu * st.capq + mv.dst) * (long long)QSLOT;
    uint8_t* hs = st.hstore + (gu * st.caps + mv.sent) * (long long)BSLOT;
    cp_async_wait_all_but_newest();
    __syncthreads();
    if (mv.kind == MOVE_PACK_COPY)
      for (int o = tid * 16; o < BSLOT; o += MOVE_THREADS * 16)
        *reinterpret_cast<uint4*>(hs + o) = *reinterpret_cast<const uint4*>(raw + o);
    const int lo = (mv.win == 0) ? st.n_sink : 0;
    // key groups: one per channel over rows [lo, W), TPC threads per channel
    {
      constexpr int TPC = MOVE_THREADS / D;
      const int c = tid / TPC, part = tid % TPC;
      float mn = INFINITY, mx = -INFINITY;
      for (int r = lo + part; r < W; r += TPC) {
        const float x = bf16_at(raw, bf16_k_off(g, r, c));
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
#pragma unroll
      for (int o = 1; o < TPC; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      const float sc = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
      float T[3];
      group_thresholds<TPC>(sc, part, T);
      if (part == 0) {
        kz[c] = mn;
        ks[c] = sc;
        kp[c] = make_float4(mn, T[0], T[1], T[2]);
      }
    }
    // value groups: one per token over D channels; 8 threads per token, shuffle-reduced
#pragma unroll
    for (int t0 = 0; t0 < W; t0 += MOVE_THREADS / 8) {
      const int r = t0 + tid / 8, part = tid % 8;
      float mn = INFINITY, mx = -INFINITY;
      if (r < W) {
        for (int c = part; c < D; c += 8) {
          const float x = bf16_at(raw, bf16_v_off(g, r, c));
          mn = fminf(mn, x);
          mx = fmaxf(mx, x);
        }
      }
#pragma unroll
      for (int o = 4; o; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      const bool sink = r < lo;
      const float sc = sink ? 0.f : __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
      float T[3];
      group_thresholds<8>(r < W ? sc : 0.f, part, T);
      if (r < W && part == 0) {
        vz[r] = sink ? 0.f : mn;
        vs[r] = sc;
        vp[r] = make_float4(sink ? 0.f : mn, T[0], T[1], T[2]);
      }
    }
    __syncthreads();
    // codes: each thread assembles whole 32-bit words.  Word (lane, wi) of a code block holds
    // fragments 2 wi and 2 wi + 1 of that lane; the bf16 slot stores the same fragment of the
    // same lane as one 16-byte vector (element (reg, e) at bits 32 reg + 16 e), so a word needs
    // two vector loads and its code (reg, f, e) goes to bit 8 f + 2 reg + 16 e.
    constexpr int WPL = (W / 16) * (D / 16) / 2, CW = WPL < 4 ? WPL : 4, KS = D / 16, KT = W / 16;
    constexpr int SUB = 64 * D, OFF_VCODE = W * D / 4 + 8 * D;
#pragma unroll
    for (int t = tid; t < 64 * WPL; t += MOVE_THREADS) {
      const bool value = t >= 32 * WPL;
      const int tt = value ? t - 32 * WPL : t;
      const int lane = tt & 31, wi = tt >> 5;
      const int widx = ((wi / CW) * 32 + lane) * CW + (wi % CW);
      const int a = lane >> 2, b = 2 * (lane & 3);
      unsigned word = 0u;
#pragma unroll
      for (int f = 0; f < 2; ++f) {
        const int F = 2 * wi + f;
        uint4 x;
        int r0, c0;   // row / column of element (reg 0, e 0) of this lane's fragment
        if (!value) {
          const int mt = F / KS, kst = F % KS;
          x = *reinterpret_cast<const uint4*>(raw + mt * SUB + kst * 512 + lane * 16);
          r0 = 16 * mt + a;
          c0 = 16 * kst + b;
        } else {
          const int mc = F / KT, kt = F % KT;
          x = *reinterpret_cast<const uint4*>(raw + kt * SUB + 32 * D + mc * 512 + lane * 16);
          r0 = 16 * kt + b;   // token
          c0 = 16 * mc + a;   // channel
        }
        const unsigned xr[4] = {x.x, x.y, x.z, x.w};
        if (!value) {
          // channels c0, c0 + 1, c0 + 8, c0 + 9; rows r0, r0 + 8
#pragma unroll
          for (int hc = 0; hc < 2; ++hc)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = c0 + e + 8 * hc;
              const float4 pc = kp[c];
              const float sc = ks[c];
#pragma unroll
              for (int hr = 0; hr < 2; ++hr) {
                const int reg = hr + 2 * hc;
                const float xv = __uint_as_float(e ? (xr[reg] & 0xFFFF0000u) : (xr[reg] << 16));
                const unsigned code = r0 + 8 * hr >= lo ? quant_code(xv, pc, sc) : 0u;
                word |= code << (8 * f + 2 * reg + 16 * e);
              }
            }
        } else {
          // tokens r0, r0 + 1, r0 + 8, r0 + 9; channels c0, c0 + 8
#pragma unroll
          for (int hr = 0; hr < 2; ++hr)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int r = r0 + e + 8 * hr;
              const float4 pr = vp[r];
              const float sr = vs[r];
#pragma unroll
              for (int hc = 0; hc < 2; ++hc) {
                const int reg = hc + 2 * hr;
                const float xv = __uint_as_float(e ? (xr[reg] & 0xFFFF0000u) : (xr[reg] << 16));
                const unsigned code = r >= lo ? quant_code(xv, pr, sr) : 0u;
                word |= code << (8 * f + 2 * reg + 16 * e);
              }
            }
        }
      }
      const int wo = (value ? OFF_VCODE / 4 : 0) + widx;
      reinterpret_cast<unsigned*>(qimg)[wo] = word;
    }
    for (int c = tid; c < D; c += MOVE_THREADS) {
      const int pc = kparam_pos(c);
      reinterpret_cast<float*>(qimg + g.off_kmin())[pc] = kz[c];
      reinterpret_cast<float*>(qimg + g.off_kscale())[pc] = ks[c];
    }
    for (int r = tid; r < W; r += MOVE_THREADS) {
      const int pr = vparam_pos(g, r);
      reinterpret_cast<float*>(qimg + g.off_vmin())[pr] = vz[r];
      reinterpret_cast<float*>(qimg + g.off_vscale())[pr] = vs[r];
    }
    if (tid < 32) write_qrange(st, gu, mv.dst, ks, vs, D, W, tid);
    __syncthreads();
    // the slot in whole 16-byte vectors; its codes reach the host ledger only if the slot is
    // later handed to another window while this one is still kept (the write-back above)
    for (int o = tid * 16; o < QSLOT; o += MOVE_THREADS * 16)
      *reinterpret_cast<uint4*>(qs + o) = *reinterpret_cast<const uint4*>(qimg + o);
    __syncthreads();   // shared memory is reused by this CTA's next move
  }
}

// ------------------------------------------------------------------------------ launchers
// Commit of a speculative verify of n_q draft tokens from length L0 (H2O page §5, speculative
// decoding): drafts [n_accept, n_q) are dropped -- the windows they opened close in reverse
// opening order (their bf16 slots go back to the free list's head, from which they were taken;
// the slot no longer holds an evicted window's exact data) -- and the accepted queries' window
// masses are added to the scores in query order.  CTAs (unit, y): y = 0 closes the dropped
// drafts' windows (all of them at or past the new window count), every y adds the masses of a
// quarter of the kept windows; block (0, 0) sets the length.
constexpr int VCOMMIT_SPLIT = 4;
__global__ void __launch_bounds__(256) qe_verify_commit_kernel(State st, int layer, int L0, int n_q, int n_accept,
                                                               const float* delta, long long qstride) {
  const int u = blockIdx.x, y = blockIdx.y;
  const long long gu = (long long)layer * st.units + u;
  const int W = st.geo.W;
  const int new_L = L0 + n_accept, old_L = L0 + n_q;
  const int first_opened = (L0 + W - 1) / W;             // windows starting at or after L0
  const int new_nwin = (new_L + W - 1) / W, old_nwin = (old_L + W - 1) / W;
  if (y == 0 && threadIdx.x == 0) {
    for (int j = old_nwin - 1; j >= new_nwin && j >= first_opened; --j) {
      const int s = st.bslot[gu * st.maxw + j];
      const int head = st.bfree_head[gu] - 1;
      if (s < 0 || s >= st.capb || head < 0 || st.bfree[gu * st.capb + head] != s) {
        atomicOr(st.err, ERR_FREELIST);
        break;
      }
      st.bfree_head[gu] = head;
      st.bvictim[gu * st.capb + s] = -1;
      st.bslot[gu * st.maxw + j] = -1;
      st.tier[gu * st.maxw + j] = TIER_NONE;
      st.score[gu * st.maxw + j] = 0.f;
    }
  }
  const int j0 = (int)((long long)y * new_nwin / VCOMMIT_SPLIT), j1 = (int)((long long)(y + 1) * new_nwin / VCOMMIT_SPLIT);
  for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
    const float* dj = delta + (long long)u * st.maxw + j;
    float sc = st.score[gu * st.maxw + j];
    for (int q = 0; q < n_accept; ++q) sc += dj[q * qstride];
    st.score[gu * st.maxw + j] = sc;
  }
  if (u == 0 && y == 0 && threadIdx.x == 0) st.ldev[layer].L = new_L;
}

cudaError_t launch_verify_commit(const State& st, int layer, int L0, int n_q, int n_accept, const float* delta,
                                 long long qstride, cudaStream_t s) {
  qe_verify_commit_kernel<<<dim3(st.units, VCOMMIT_SPLIT), 256, 0, s>>>(st, layer, L0, n_q, n_accept, delta, qstride);
  return cudaGetLastError();
}

cudaError_t launch_append(const State& st, int layer, int n, const uint16_t* k, const uint16_t* v, int n_sm,
                          cudaStream_t s, bool tok_major) {
  if (n == 1 && !tok_major) {
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
  qe_append_kernel<<<(int)blocks, 256, 0, s>>>(st, layer, n, k, v, tok_major ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_commit_length(const State& st, int layer, int n, cudaStream_t s) {
  qe_commit_length_kernel<<<1, 1, 0, s>>>(st, layer, n);
  return cudaGetLastError();
}

size_t route_smem_bytes(const State& st) {
  const int cc = route_cand_cap(st);
  return (size_t)route_key_cap(st) * 8 + (size_t)cc * 4 * 6 + (size_t)((cc + 15) & ~15) * 2 +
         (size_t)(3 * st.capb + 4 * st.capq + st.caps) * 4 + (size_t)(st.capb + st.capq) + 16;
}

cudaError_t launch_route(const RouteParams& p, int n_layers, cudaStream_t s) {
  qe_route_kernel<<<dim3(p.st.units, n_layers), ROUTE_THREADS, route_smem_bytes(p.st), s>>>(p);
  return cudaGetLastError();
}

size_t move_smem_bytes(const State& st) {
  const int W = st.geo.W, D = st.geo.D;
  return (size_t)2 * st.geo.bslot_bytes() + (size_t)(D + W) * (16 + 8) + (size_t)st.geo.qslot_bytes();
}

// the move kernel of a geometry (head_dim 64 or 128, window 16, 32 or 64), or null
using MoveKernel = void (*)(State, const Move*, const int*);
static MoveKernel move_kernel_for(int D, int W) {
  if (D == 128) return W == 16 ? qe_move_kernel<128, 16> : W == 32 ? qe_move_kernel<128, 32> : W == 64 ? qe_move_kernel<128, 64> : nullptr;
  if (D == 64) return W == 16 ? qe_move_kernel<64, 16> : W == 32 ? qe_move_kernel<64, 32> : W == 64 ? qe_move_kernel<64, 64> : nullptr;
  return nullptr;
}

cudaError_t launch_moves(const State& st, const Move* moves, const int* n_moves, int n_sm, cudaStream_t s) {
  const MoveKernel k = move_kernel_for(st.geo.D, st.geo.W);
  if (!k) return cudaErrorInvalidValue;
  k<<<n_sm * MOVE_CTAS_PER_SM, MOVE_THREADS, move_smem_bytes(st), s>>>(st, moves, n_moves);
  return cudaGetLastError();
}

// kernel attributes, set once (outside any stream capture)
// The limit is a property of the kernel, shared by every handle of the process: it is raised to
// the device's opt-in maximum (never lowered for a smaller handle), and a handle whose routing
// needs more is refused.
cudaError_t prepare_route_kernels(const State& st) {
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const MoveKernel mk = move_kernel_for(st.geo.D, st.geo.W);
  if (!mk) return cudaErrorInvalidValue;
  cudaFuncAttributes ra{}, ma{};
  if ((e = cudaFuncGetAttributes(&ra, qe_route_kernel)) != cudaSuccess) return e;
  if ((e = cudaFuncGetAttributes(&ma, mk)) != cudaSuccess) return e;
  const int rmax = optin - (int)ra.sharedSizeBytes, mmax = optin - (int)ma.sharedSizeBytes;
  if (route_smem_bytes(st) > (size_t)rmax || move_smem_bytes(st) > (size_t)mmax) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(qe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, rmax);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mk, cudaFuncAttributeMaxDynamicSharedMemorySize, mmax);
}

}  // namespace qe
