// qe_attn.cu -- qe_decode_attn (split-K flash-decode over bf16 and 2-bit tiles with fused
// per-window score partials) and qe_attn_combine (split merge, output, score update).
//
// What it computes (QEvict reading notes, §4.1 eq. "attention"; §4.2 eq. (1); H2O page,
// §5.1 GQA group sum): for every unit (batch element, KV head) and its G query heads,
// o_h = softmax(q_h K_acc^T / sqrt(d)) V_acc over the sink, the Pinned/Full bf16 windows
// and the 2-bit windows dequantized as x = code * s + z (HqeKV reading notes, §2.3 eq. (2);
// keys with per-channel min/scale, values with per-token min/scale), and the mass each
// window receives summed over the G heads, added to the window's float32 score.
//
// GB300 design:
//  * One persistent CTA per SM, 8 independent consumer warps.  The unit x tile sequence of
//    the layer is cut into one contiguous, cost-weighted range per warp (stream-K), so every
//    warp streams its own range through a private ring of shared-memory stages filled by
//    cp.async.bulk (one 1-D bulk copy per tile, completion on an mbarrier), and the whole GPU
//    is busy until the last tile regardless of how units and tiles divide.
//  * The G query heads of a KV head share every K/V element: the Q K^T and P V products are
//    small dense contractions ([16 tokens x d] x [d x 8]) run on the tensor cores with
//    mma.m16n8k16 (bf16 in, fp32 accumulate).  The 8 columns hold the G heads twice, as a
//    bf16 "hi" part and a bf16 "lo" remainder of the fp32 operand (q * s_K for 2-bit keys,
//    p or p * s_V for the values), so the products keep ~16 bits of operand precision.
//  * 2-bit codes are unpacked in registers straight into mma fragments (the slots are stored
//    in fragment order), never materialised as bf16 in memory.
//  * Per-window mass leaves the kernel as a log-sum-exp per (tile, head); the combine kernel
//    turns it into a probability mass once the unit's global softmax normaliser is known.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qe_kernels.cuh"

namespace qe {

constexpr int ATTN_WARPS = 8;
constexpr int ATTN_SMEM_STAGES_BYTES = 196608;   // 192 KB of stages per CTA
constexpr unsigned long long WAIT_LIMIT_NS = 200000000ull;  // 0.2 s

struct TileDesc {
  int u, i;        // unit, tile index in unit
  int slot, win;   // slot in its pool, window id (-1 for the sink)
  int lo, hi;      // valid rows inside the tile
  int kind;        // 0 bf16 sub-tile, 1 2-bit window
  int pad;
};

__device__ __forceinline__ long long tile_start(const AttnParams& p, int u, int i, int nbt) {
  long long r = (i < nbt) ? (long long)i * p.cb : (long long)nbt * p.cb + (long long)(i - nbt) * p.cq;
  return (long long)u * p.Cu + r;
}

// first tile whose start position is >= x
__device__ __forceinline__ void first_tile(const AttnParams& p, long long x, int nbt, int& u, int& i) {
  u = (int)(x / p.Cu);
  long long r = x - (long long)u * p.Cu;
  long long bend = (long long)nbt * p.cb;
  if (r <= (long long)(nbt - 1) * p.cb) {
    i = (int)((r + p.cb - 1) / p.cb);
  } else if (p.nq > 0 && r <= bend) {
    i = nbt;                                   // between the last bf16 tile and the first 2-bit one
  } else if (p.nq > 0 && r <= bend + (long long)(p.nq - 1) * p.cq) {
    i = nbt + (int)((r - bend + p.cq - 1) / p.cq);
  } else {
    u += 1;
    i = 0;
  }
}

// fill the descriptor of (u, i); returns false if the tile has no valid row
__device__ __forceinline__ bool describe(const AttnParams& p, int u, int i, int nbt, TileDesc& d) {
  const State& st = p.st;
  const int W = st.geo.W;
  const int sub_tiles = W / 16;
  const long long gu = (long long)p.layer * st.units + u;
  d.u = u;
  d.i = i;
  if (i < nbt) {
    int e = i / sub_tiles, sub = i - e * sub_tiles;
    int2 ent = st.blist[gu * st.capb + e];
    d.win = ent.x;
    d.slot = ent.y;
    d.kind = 0;
    if (ent.y < 0 || ent.y >= st.capb || ent.x < -1 || ent.x >= st.maxw) {   // corrupt entry: skip, flag
      atomicOr(st.err, ERR_TABLE);
      return false;
    }
    int lo, hi;
    if (ent.x < 0) {
      lo = 0;
      hi = st.n_sink;
    } else {
      lo = (ent.x == 0) ? st.n_sink : 0;
      int h = p.L - ent.x * W;
      hi = h < W ? h : W;
    }
    int base = sub * 16;
    int tl = lo - base, th = hi - base;
    d.lo = tl < 0 ? 0 : tl;
    d.hi = th > 16 ? 16 : th;
    d.pad = sub;
    return d.hi > d.lo;
  }
  int2 ent = st.qlist[gu * st.capq + (i - nbt)];
  d.win = ent.x;
  d.slot = ent.y;
  d.kind = 1;
  if (ent.y < 0 || ent.y >= st.capq || ent.x < 0 || ent.x >= st.maxw) {
    atomicOr(st.err, ERR_TABLE);
    return false;
  }
  d.lo = (ent.x == 0) ? st.n_sink : 0;
  d.hi = W;
  d.pad = 0;
  return true;
}

__device__ __forceinline__ const uint8_t* tile_src(const AttnParams& p, const TileDesc& d, unsigned& bytes) {
  const State& st = p.st;
  const long long gu = (long long)p.layer * st.units + d.u;
  if (d.kind == 0) {
    bytes = st.geo.sub_bytes();
    return st.bslab + ((gu * st.capb + d.slot) * (long long)st.geo.bslot_bytes()) + (long long)d.pad * st.geo.sub_bytes();
  }
  bytes = st.geo.qslot_bytes();
  return st.qslab + (gu * st.capq + d.slot) * (long long)st.geo.qslot_bytes();
}

// Advance (u, i) to the next tile in sequence order.
__device__ __forceinline__ void next_tile(const AttnParams& p, int& u, int& i) {
  i += 1;
  if (i >= p.ntiles) {
    i = 0;
    u += 1;
  }
}

template <int D, int W>
struct Shape {
  static constexpr int KS = D / 16;
  static constexpr int MC = D / 16;
  static constexpr int MT = W / 16;
  static constexpr int KT = W / 16;
  static constexpr int WPL = MT * KS / 2;
  static constexpr int CW = WPL < 4 ? WPL : 4;
  static constexpr int SUB_BYTES = 64 * D;
  static constexpr int QSLOT = 2 * (W * D / 4) + 8 * D + 8 * W;
  static constexpr int STAGE = SUB_BYTES > QSLOT ? SUB_BYTES : QSLOT;
  static constexpr int NST = ATTN_SMEM_STAGES_BYTES / (ATTN_WARPS * STAGE);
  static constexpr int KCODE = W * D / 4;
  static constexpr int OFF_KMIN = 2 * KCODE;
  static constexpr int OFF_KSCALE = 2 * KCODE + 4 * D;
  static constexpr int OFF_VMIN = 2 * KCODE + 8 * D;
  static constexpr int OFF_VSCALE = 2 * KCODE + 8 * D + 4 * W;
};

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// Load this lane's code words (WPL of them) of one code block.
template <int WPL, int CW>
__device__ __forceinline__ void load_words(const uint8_t* blk, int lane, unsigned (&w)[WPL]) {
#pragma unroll
  for (int c = 0; c < WPL / CW; ++c) {
    const uint8_t* src = blk + (c * 32 + lane) * (CW * 4);
    if constexpr (CW == 4) {
      uint4 v = lds128(src);
      w[c * 4 + 0] = v.x; w[c * 4 + 1] = v.y; w[c * 4 + 2] = v.z; w[c * 4 + 3] = v.w;
    } else if constexpr (CW == 2) {
      uint2 v = *reinterpret_cast<const uint2*>(src);
      w[c * 2 + 0] = v.x; w[c * 2 + 1] = v.y;
    } else {
      w[c] = *reinterpret_cast<const unsigned*>(src);
    }
  }
}

// Online-softmax step over one tile of MT m-tiles whose Q K^T accumulators are in acc.
// Produces the P^T B-fragments (hi/lo split) for the P V product, updates (m, l, zsum, O).
template <int MT, int MC, bool INT2>
__device__ __forceinline__ void softmax_tile(float (&acc)[MT][4], int lo, int hi, const float (&bias)[2],
                                             const float* vmin, const float* vscale, float scale_log2,
                                             float (&m)[2], float (&l)[2], float (&zs)[2], float (&O)[MC][4],
                                             unsigned (&Bp)[MT][2], float* lse_out, int G, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float x[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float v = acc[mt][r] + __shfl_xor_sync(0xffffffffu, acc[mt][r], 2);
      int row = mt * 16 + g + ((r & 2) ? 8 : 0);
      v = (v + bias[r & 1]) * scale_log2;
      x[mt][r] = (row >= lo && row < hi) ? v : -INFINITY;
    }
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) mx[r & 1] = fmaxf(mx[r & 1], x[mt][r]);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
    mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
    mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
  }
  float mnew[2], muse[2], alpha[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    mnew[e] = fmaxf(m[e], mx[e]);
    muse[e] = (mnew[e] == -INFINITY) ? 0.f : mnew[e];
    alpha[e] = ex2(m[e] - muse[e]);
  }
  float pr[MT][4];
  float mass[2] = {0.f, 0.f};
  float zadd[2] = {0.f, 0.f};
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float pv = ex2(x[mt][r] - muse[r & 1]);
      pr[mt][r] = pv;
      mass[r & 1] += pv;
      if constexpr (INT2) {
        int row = mt * 16 + g + ((r & 2) ? 8 : 0);
        zadd[r & 1] = fmaf(pv, vmin[row], zadd[r & 1]);
      }
    }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    mass[e] += __shfl_xor_sync(0xffffffffu, mass[e], 4);
    mass[e] += __shfl_xor_sync(0xffffffffu, mass[e], 8);
    mass[e] += __shfl_xor_sync(0xffffffffu, mass[e], 16);
    l[e] = fmaf(l[e], alpha[e], mass[e]);
    zs[e] = fmaf(zs[e], alpha[e], zadd[e]);
    m[e] = mnew[e];
  }
  // per-tile log2-sum-exp of each head (heads 2t, 2t+1 written by lanes 0 and 1)
  if (lse_out != nullptr && g == 0 && t < 2) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int h = 2 * t + e;
      if (h < G) lse_out[h] = mass[e] > 0.f ? muse[e] + lg2(mass[e]) : -INFINITY;
    }
  }
#pragma unroll
  for (int mc = 0; mc < MC; ++mc)
#pragma unroll
    for (int r = 0; r < 4; ++r) O[mc][r] *= alpha[r & 1];
  // P^T fragments: columns 0..3 carry the bf16 "hi" part of each head, 4..7 the remainder
  const bool lo_lane = t >= 2;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    float y[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float v = pr[mt][r];
      if constexpr (INT2) {
        int row = mt * 16 + g + ((r & 2) ? 8 : 0);
        v *= vscale[row];
      }
      y[r] = v;
    }
    unsigned top, bot;
    {
      unsigned y0 = __float_as_uint(y[0]), y1 = __float_as_uint(y[1]);
      unsigned y2 = __float_as_uint(y[2]), y3 = __float_as_uint(y[3]);
      unsigned h01 = __byte_perm(y0, y1, 0x7632), h23 = __byte_perm(y2, y3, 0x7632);
      unsigned l01 = pack_bf16x2(y[0] - __uint_as_float(y0 & 0xFFFF0000u), y[1] - __uint_as_float(y1 & 0xFFFF0000u));
      unsigned l23 = pack_bf16x2(y[2] - __uint_as_float(y2 & 0xFFFF0000u), y[3] - __uint_as_float(y3 & 0xFFFF0000u));
      top = lo_lane ? l01 : h01;
      bot = lo_lane ? l23 : h23;
    }
    Bp[mt][0] = movmatrix_t(top);
    Bp[mt][1] = movmatrix_t(bot);
  }
}

template <int D, int W>
__global__ void __launch_bounds__(ATTN_WARPS * 32, 1) qe_decode_attn_kernel(const AttnParams p) {
  using S = Shape<D, W>;
  constexpr int KS = S::KS, MC = S::MC, MT = S::MT, KT = S::KT, WPL = S::WPL, CW = S::CW, NST = S::NST;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) unsigned long long bars[ATTN_WARPS][NST];
  __shared__ TileDesc descs[ATTN_WARPS][NST];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.st.G;
  const int wg = blockIdx.x * ATTN_WARPS + warp;
  const long long x_lo = (wg * p.C + p.NW - 1) / p.NW;
  const long long x_hi = ((wg + 1) * p.C + p.NW - 1) / p.NW;
  if (x_lo >= x_hi) return;
  const int nbt = p.nbw * (W / 16);
  const int u_first = (int)(x_lo / p.Cu);
  const int u_last = (int)((x_hi - 1) / p.Cu);

  uint8_t* stage_base = smem + (size_t)warp * NST * S::STAGE;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
    mbar_fence_init();
  }
  __syncwarp();

  // producer cursor
  int pu, pi;
  first_tile(p, x_lo, nbt, pu, pi);
  int issued = 0;
  auto issue_next = [&](int slot_stage) -> bool {
    // advance the producer cursor to the next non-empty tile inside the range
    while (pu < p.st.units && tile_start(p, pu, pi, nbt) < x_hi) {
      TileDesc d;
      bool ok = describe(p, pu, pi, nbt, d);
      next_tile(p, pu, pi);
      if (!ok) continue;
      if (lane == 0) {
        descs[warp][slot_stage] = d;
        unsigned bytes;
        const uint8_t* src = tile_src(p, d, bytes);
        unsigned bar = smem_u32(&bars[warp][slot_stage]);
        mbar_expect_tx(bar, bytes);
        bulk_g2s(smem_u32(stage_base + (size_t)slot_stage * S::STAGE), src, bytes, bar);
      }
      return true;
    }
    return false;
  };
  int n_inflight = 0;
  for (int s = 0; s < NST; ++s) {
    if (!issue_next(s)) break;
    ++n_inflight;
    ++issued;
  }
  __syncwarp();

  // consumer state of the current unit
  float m[2], l[2], zs[2];
  float O[MC][4];
  unsigned qv[KS][2];      // this lane's head (g & 3) query values, bf16 pairs
  unsigned qb[KS][2];      // B fragments for bf16 tiles (zero in lo columns)
  int cur_u = u_first;
  int q_unit = -1;
  auto reset = [&]() {
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
    zs[0] = zs[1] = 0.f;
#pragma unroll
    for (int mc = 0; mc < MC; ++mc)
#pragma unroll
      for (int r = 0; r < 4; ++r) O[mc][r] = 0.f;
  };
  auto flush = [&](int u) {
    const long long pidx = (long long)wg * p.maxseg + (u - u_first);
    // O^T[c][n]: add the lo column (n + 4) to the hi column n; add the value-bias term
    float zt[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float z = zs[e];
      z += __shfl_xor_sync(0xffffffffu, z, 4);
      z += __shfl_xor_sync(0xffffffffu, z, 8);
      z += __shfl_xor_sync(0xffffffffu, z, 16);
      zt[e] = z;   // lanes t < 2 hold the sum over all rows for heads 2t, 2t+1
    }
#pragma unroll
    for (int mc = 0; mc < MC; ++mc)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float v = O[mc][r] + __shfl_xor_sync(0xffffffffu, O[mc][r], 2);
        int h = 2 * t + (r & 1);
        int c = mc * 16 + g + ((r & 2) ? 8 : 0);
        if (t < 2 && h < G) p.part_o[(pidx * G + h) * D + c] = v + zt[r & 1];
      }
    if (g == 0 && t < 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int h = 2 * t + e;
        if (h < G) p.part_ml[pidx * G + h] = make_float2(m[e], l[e]);
      }
    }
  };
  reset();

  const int hh = g & 3;
  const bool lo_lane_b = g >= 4;
  // bounded wait for the bulk copy of the k-th tile (false: gave up after WAIT_LIMIT_NS)
  auto wait_tile = [&](int k) -> bool {
    const unsigned bar = smem_u32(&bars[warp][k % NST]);
    const unsigned parity = (k / NST) & 1;
    unsigned long long t0 = 0;
    int spins = 0;
    bool ok = true;
    while (!mbar_try_wait(bar, parity)) {
      if (++spins == 64) {
        spins = 0;
        const unsigned long long now = globaltimer_ns();
        if (t0 == 0) t0 = now;
        else if (now - t0 > WAIT_LIMIT_NS) { ok = false; break; }
      }
    }
    return __all_sync(0xffffffffu, ok);
  };
  bool timed_out = false;
  int k = 0;
  for (; k < issued; ++k) {
    const int s = k % NST;
    if (!wait_tile(k)) { timed_out = true; break; }
    const TileDesc d = descs[warp][s];
    const uint8_t* sp = stage_base + (size_t)s * S::STAGE;
    while (d.u > cur_u) {
      flush(cur_u);
      reset();
      ++cur_u;
    }
    if (q_unit != cur_u) {
      q_unit = cur_u;
      const int b = cur_u / p.st.Hkv, kvh = cur_u - b * p.st.Hkv;
      const uint16_t* qh = p.q + ((size_t)b * p.st.Hq + kvh * G + hh) * D;
      const bool act = hh < G;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        unsigned a0 = act ? *reinterpret_cast<const unsigned*>(qh + ks * 16 + 2 * t) : 0u;
        unsigned a1 = act ? *reinterpret_cast<const unsigned*>(qh + ks * 16 + 8 + 2 * t) : 0u;
        qv[ks][0] = a0;
        qv[ks][1] = a1;
        qb[ks][0] = lo_lane_b ? 0u : a0;
        qb[ks][1] = lo_lane_b ? 0u : a1;
      }
    }
    float* lse_out = p.lse + ((size_t)d.u * p.ntiles + d.i) * G;
    if (d.kind == 0) {
      // ---- bf16 sub-tile: 16 tokens
      float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint4 a = lds128(sp + ks * 512 + lane * 16);
        mma_bf16(acc[0], a.x, a.y, a.z, a.w, qb[ks][0], qb[ks][1]);
      }
      const float bias[2] = {0.f, 0.f};
      unsigned Bp[1][2];
      softmax_tile<1, MC, false>(acc, d.lo, d.hi, bias, nullptr, nullptr, p.scale_log2, m, l, zs, O, Bp, lse_out, G,
                                 lane);
#pragma unroll
      for (int mc = 0; mc < MC; ++mc) {
        uint4 a = lds128(sp + 32 * D + mc * 512 + lane * 16);
        mma_bf16(O[mc], a.x, a.y, a.z, a.w, Bp[0][0], Bp[0][1]);
      }
    } else {
      // ---- 2-bit window: W tokens
      const float* kmin = reinterpret_cast<const float*>(sp + S::OFF_KMIN);
      const float* kscale = reinterpret_cast<const float*>(sp + S::OFF_KSCALE);
      const float* vmin = reinterpret_cast<const float*>(sp + S::OFF_VMIN);
      const float* vscale = reinterpret_cast<const float*>(sp + S::OFF_VSCALE);
      // B fragments q' = q * s_K (hi part in lanes g < 4, remainder in lanes g >= 4), bias q . z_K
      unsigned qp[KS][2];
      float bpart = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int c = ks * 16 + hf * 8 + 2 * t;
          const float2 sc = *reinterpret_cast<const float2*>(kscale + c);
          const float2 zc = *reinterpret_cast<const float2*>(kmin + c);
          const float q0 = bf16lo_to_f32(qv[ks][hf]), q1 = bf16hi_to_f32(qv[ks][hf]);
          bpart = fmaf(q0, zc.x, bpart);
          bpart = fmaf(q1, zc.y, bpart);
          const float y0 = q0 * sc.x, y1 = q1 * sc.y;
          const unsigned u0 = __float_as_uint(y0), u1 = __float_as_uint(y1);
          const unsigned hi2 = __byte_perm(u0, u1, 0x7632);
          const unsigned lo2 = pack_bf16x2(y0 - __uint_as_float(u0 & 0xFFFF0000u), y1 - __uint_as_float(u1 & 0xFFFF0000u));
          qp[ks][hf] = lo_lane_b ? lo2 : hi2;
        }
      }
      bpart += __shfl_xor_sync(0xffffffffu, bpart, 1);
      bpart += __shfl_xor_sync(0xffffffffu, bpart, 2);
      float bias[2];
      bias[0] = __shfl_sync(0xffffffffu, bpart, (2 * (t & 1)) * 4);
      bias[1] = __shfl_sync(0xffffffffu, bpart, (2 * (t & 1) + 1) * 4);
      // Q K^T over the unpacked key codes
      float acc[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mt][r] = 0.f;
      {
        unsigned wk[WPL];
        load_words<WPL, CW>(sp, lane, wk);
#pragma unroll
        for (int wi = 0; wi < WPL; ++wi) {
          unsigned a[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) a[j] = codes_to_bf16x2(wk[wi] >> (2 * j));
#pragma unroll
          for (int f = 0; f < 2; ++f) {
            const int F = 2 * wi + f;
            const int mt = F / KS, ks = F % KS;
            mma_bf16(acc[mt], a[4 * f + 0], a[4 * f + 1], a[4 * f + 2], a[4 * f + 3], qp[ks][0], qp[ks][1]);
          }
        }
      }
      unsigned Bp[MT][2];
      softmax_tile<MT, MC, true>(acc, d.lo, d.hi, bias, vmin, vscale, p.scale_log2, m, l, zs, O, Bp, lse_out, G,
                                 lane);
      // P V over the unpacked value codes (A = V^T: channel tiles x token steps)
      {
        unsigned wv[WPL];
        load_words<WPL, CW>(sp + S::KCODE, lane, wv);
#pragma unroll
        for (int wi = 0; wi < WPL; ++wi) {
          unsigned a[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) a[j] = codes_to_bf16x2(wv[wi] >> (2 * j));
#pragma unroll
          for (int f = 0; f < 2; ++f) {
            const int F = 2 * wi + f;
            const int mc = F / KT, kt = F % KT;
            mma_bf16(O[mc], a[4 * f + 0], a[4 * f + 1], a[4 * f + 2], a[4 * f + 3], Bp[kt][0], Bp[kt][1]);
          }
        }
      }
    }
    __syncwarp();
    // refill this stage
    if (issue_next(s)) ++issued;
    __syncwarp();
  }
  if (timed_out) {
    // report, then give the copies still in flight a bounded chance to land before exiting
    if (lane == 0) atomicOr(p.st.err, ERR_TIMEOUT);
    for (int kk = k + 1; kk < issued; ++kk) wait_tile(kk);
    return;
  }
  while (cur_u <= u_last) {
    flush(cur_u);
    reset();
    ++cur_u;
  }
}

// ------------------------------------------------------------------------------ combine
// One CTA per unit: merge the partials of every warp whose range meets the unit, write
// o = sum / l, then turn each tile's log2-sum-exp into mass, sum it over the G heads and
// add it to the window's float32 score (eq. (1) with the GQA group sum).
template <int D>
__global__ void __launch_bounds__(128) qe_attn_combine_kernel(const CombineParams p) {
  const int u = blockIdx.x;
  const int G = p.st.G;
  const long long gu = (long long)p.layer * p.st.units + u;
  constexpr int MAXP = 256;
  __shared__ float s_M[4], s_scale[4 * MAXP], s_lse[4];
  __shared__ int s_np;
  __shared__ long long s_pidx[MAXP];
  // partial producers: warps whose position range meets [u Cu, (u+1) Cu)
  if (threadIdx.x == 0) {
    long long a = (long long)u * p.Cu, b = a + p.Cu - 1;
    long long w0 = a * p.NW / p.C, w1 = b * p.NW / p.C;
    int np = 0;
    for (long long w = w0; w <= w1 && np < MAXP; ++w) {
      long long xl = (w * p.C + p.NW - 1) / p.NW, xh = ((w + 1) * p.C + p.NW - 1) / p.NW;
      if (xl >= xh) continue;
      s_pidx[np++] = w * p.maxseg + (u - (int)(xl / p.Cu));
    }
    if (w1 - w0 + 1 > MAXP) atomicOr(p.st.err, ERR_COUNT);
    s_np = np;
  }
  __syncthreads();
  const int np = s_np;
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = -INFINITY;
    for (int k = 0; k < np; ++k) M = fmaxf(M, p.part_ml[s_pidx[k] * G + h].x);
    float Mu = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f;
    for (int k = 0; k < np; ++k) {
      float2 ml = p.part_ml[s_pidx[k] * G + h];
      float sc = ex2(ml.x - Mu);
      s_scale[h * MAXP + k] = sc;
      Ls += ml.y * sc;
    }
    s_M[h] = Ls;
    s_lse[h] = Mu + lg2(Ls);
  }
  __syncthreads();
  const int b = u / p.st.Hkv, kvh = u - b * p.st.Hkv;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int h = e / D, c = e - h * D;
    float acc = 0.f;
    for (int k = 0; k < np; ++k) acc = fmaf(p.part_o[(s_pidx[k] * G + h) * D + c], s_scale[h * MAXP + k], acc);
    const float o = acc / s_M[h];
    const size_t oi = ((size_t)b * p.st.Hq + kvh * G + h) * D + c;
    if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = o;
    else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
  }
  // scores: bf16 window entries (skip the sink) and 2-bit windows
  const int W = p.st.geo.W, sub_tiles = W / 16;
  const int nent = p.nbw + p.nq;
  for (int e = threadIdx.x; e < nent; e += blockDim.x) {
    int win;
    float dS = 0.f;
    if (e < p.nbw) {
      int2 ent = p.st.blist[gu * p.st.capb + e];
      win = ent.x;
      if (win < 0) continue;
      int lo = (win == 0) ? p.st.n_sink : 0;
      int hi = p.L - win * W;
      hi = hi < W ? hi : W;
      for (int s = 0; s < sub_tiles; ++s) {
        int tl = lo - 16 * s, th = hi - 16 * s;
        if ((th > 16 ? 16 : th) <= (tl < 0 ? 0 : tl)) continue;
        const float* ls = p.lse + ((size_t)u * p.ntiles + e * sub_tiles + s) * G;
        for (int h = 0; h < G; ++h) dS += ex2(ls[h] - s_lse[h]);
      }
    } else {
      int2 ent = p.st.qlist[gu * p.st.capq + (e - p.nbw)];
      win = ent.x;
      const float* ls = p.lse + ((size_t)u * p.ntiles + p.nbw * sub_tiles + (e - p.nbw)) * G;
      for (int h = 0; h < G; ++h) dS += ex2(ls[h] - s_lse[h]);
    }
    if (win < 0 || win >= p.st.maxw) {
      atomicOr(p.st.err, ERR_TABLE);
      continue;
    }
    float* sp = p.st.score + gu * p.st.maxw + win;
    *sp = *sp + dS;
  }
}

// ------------------------------------------------------------------------------ launchers
template <int D, int W>
static cudaError_t launch_attn_t(const AttnParams& p, int grid, cudaStream_t stream) {
  using S = Shape<D, W>;
  const size_t smem = (size_t)ATTN_WARPS * S::NST * S::STAGE;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(qe_decode_attn_kernel<D, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  qe_decode_attn_kernel<D, W><<<grid, ATTN_WARPS * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_attn(const AttnParams& p, int grid, cudaStream_t stream) {
  const int D = p.st.geo.D, W = p.st.geo.W;
  if (D == 128 && W == 32) return launch_attn_t<128, 32>(p, grid, stream);
  if (D == 128 && W == 16) return launch_attn_t<128, 16>(p, grid, stream);
  if (D == 128 && W == 64) return launch_attn_t<128, 64>(p, grid, stream);
  if (D == 64 && W == 16) return launch_attn_t<64, 16>(p, grid, stream);
  if (D == 64 && W == 32) return launch_attn_t<64, 32>(p, grid, stream);
  if (D == 64 && W == 64) return launch_attn_t<64, 64>(p, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_combine(const CombineParams& p, cudaStream_t stream) {
  if (p.st.geo.D == 128) qe_attn_combine_kernel<128><<<p.st.units, 128, 0, stream>>>(p);
  else qe_attn_combine_kernel<64><<<p.st.units, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

int attn_warps_per_cta() { return ATTN_WARPS; }

}  // namespace qe
