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
//  * One persistent CTA per SM, 12 independent consumer warps.  The unit x tile sequence of
//    the layer is cut into one contiguous, cost-weighted range per warp (stream-K), so every
//    warp streams its own range through a private ring of shared-memory stages filled by
//    cp.async.bulk (one 1-D bulk copy per tile, completion on an mbarrier), and the whole GPU
//    is busy until the last tile regardless of how units and tiles divide.  The copies carry an
//    evict-first L2 policy: the tiles are read once per step and the cache is many times the
//    L2, so they must not push out what every step reuses (lists, partials, queries, code).
//  * Launch start: the range arithmetic is exact 32-bit integer work (qe_partition.cuh), a
//    warp's first tile is found by one 32-lane test around its estimate, and the range's first
//    copies leave before the 2-bit slots' range records are loaded.
//  * The G query heads of a KV head share every K/V element: the Q K^T and P V products are
//    small dense contractions ([16 tokens x d] x [d x 8]) run on the tensor cores with
//    mma.m16n8k16 (fp32 accumulate).  Column 2h carries head h's operand truncated to the
//    input precision ("hi"), column 2h+1 the exact remainder ("lo"), so the products keep
//    ~16 (bf16 tiles) or ~22 (2-bit tiles, f16) bits of operand precision; each lane then owns
//    one head (its accumulator pair is that head's hi and lo), so the softmax needs no
//    cross-lane merging and no lane duplicates another's work.
//  * 2-bit codes are unpacked in registers straight into mma fragments (the slots are stored
//    in fragment order): one shift and one and-or turn a register's two codes into the f16 pair
//    (1 + code / 4).  The factor 4 goes into the logit scale (keys) and the B operand
//    (4 p s_V for values); the constant 1 into the key bias (q . (z_K / 4 - s_K)) and the value
//    offset (p . (z_V - 4 s_V)).  Dequantized values never exist in memory.
//  * Magnitudes: f16 holds those products while |q| s_K < 2^15 and 2^-13 <= s_V < 2^5.  Each
//    2-bit slot carries a record of its largest key scale and its largest and smallest value
//    scales (written when the slot receives codes); a tile whose record, with the unit's largest
//    query, says otherwise takes bf16 operands: the key products as three exact bf16 parts in
//    two mma passes, the value products as bf16 truncated + remainder.
//  * Keys stored pre-RoPE are rotated in float32 and meet the query as tf32 truncated +
//    remainder parts (m16n8k8; tf32 keeps float32's exponent range, the bf16 query is exact),
//    so no key or query magnitude leaves the operand format.
//  * Per-window mass leaves the kernel as a log-sum-exp per (tile, head); the combine kernel
//    turns it into a probability mass once the unit's global softmax normaliser is known.
#include <cstdint>
#include <vector>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qe_kernels.cuh"
#include "qe_partition.cuh"

namespace qe {

constexpr int ATTN_WARPS = 12;
constexpr int ATTN_SMEM_STAGES_BYTES = 196608;   // 192 KB of stages per CTA
constexpr unsigned long long WAIT_LIMIT_NS = 200000000ull;  // 0.2 s

struct TileDesc {
  int u, i;        // unit, tile index in unit
  int slot, win;   // slot in its pool, window id (-1 for the sink)
  int lo, hi;      // valid rows inside the tile
  int kind;        // 0 bf16 sub-tile, 1 2-bit window
  int sub;         // bf16 sub-tile index inside its window slot
  int range;       // 2-bit window: its slot's range record (qrange_word)
};

// What the consumer needs of a tile (written per stage by the producer lane).
struct StageDesc {
  int u;           // unit
  int lse_off;     // (u * ntiles + i) * G
  int meta;        // lo | hi << 8 | kind << 16
  int pad;
};

// A tile ready to issue: its source and its consumer descriptor.
struct BatchDesc {
  const uint8_t* src;
  unsigned bytes;
  StageDesc sd;
  int pad;
};
constexpr int BATCH = 32;

// Step-dependent counts of the layer being processed, read from the device-resident header.
struct Lay {
  int L, nbw, nq, nbt, ntiles, NW;
  long long Cu, C;   // cost of one unit, of the layer
};
__device__ __forceinline__ Lay make_lay(const State& st, int layer, int pend, int cb, int cq, int NW) {
  LayerDev h = st.ldev[layer];
  h.L += pend;
  const LayerView v = layer_view(st.geo, h);
  Lay y;
  y.L = v.L;
  y.nbw = v.nbw;
  y.nq = v.nq;
  y.nbt = v.nbw * (st.geo.W / 16);
  y.ntiles = y.nbt + y.nq;
  y.Cu = (long long)y.nbt * cb + (long long)y.nq * cq;
  y.C = y.Cu * st.units;
  y.NW = NW;
  return y;
}

// Tile order inside a unit: the bf16 sub-tiles and the 2-bit windows are interleaved evenly
// (qe_partition.cuh), so every warp's range mixes memory-bound bf16 tiles with compute-bound
// 2-bit tiles and the SM's warps overlap the two instead of splitting into bf16 warps and
// 2-bit warps.
__device__ __forceinline__ int q_before(const Lay& y, int i) {   // 2-bit tiles among [0, i)
  return tiles_q_before(i, y.nq, y.ntiles);
}
__device__ __forceinline__ long long tile_start_in(const AttnParams& p, const Lay& y, int i) {
  return tile_cost_start(i, y.nq, y.ntiles, p.cb, p.cq);
}
__device__ __forceinline__ long long tile_start(const AttnParams& p, const Lay& y, int u, int i) {
  return (long long)u * y.Cu + tile_start_in(p, y, i);
}

// First tile whose start position is >= u Cu + r (0 <= r <= Cu); warp-collective.  Tile i starts
// less than |cb - cq| from i Cu / n (n = ntiles), so the answer lies next to floor(r n / Cu): the
// lanes test the 32 tiles around that estimate at once (a binary search takes the rare case in
// which they do not bracket it).
__device__ __forceinline__ void first_tile(const AttnParams& p, const Lay& y, int u0, long long r, int lane, int& u,
                                           int& i) {
  u = u0;
  const int n = y.ntiles;
  // P(c): c >= n, or tile c starts at or after r (false below 0); the answer is the smallest c with P
  auto P = [&](int c) -> bool { return c >= n || (c >= 0 && tile_start_in(p, y, c) >= r); };
  const int c0 = (int)first_tile_estimate(r, n, y.Cu) - 15;
  const unsigned b = __ballot_sync(0xffffffffu, P(c0 + lane));
  if (b != 0u && (!(b & 1u) || c0 == 0)) {
    i = c0 + __ffs(b) - 1;
  } else {
    int lo = 0, hi = n;   // smallest c in [0, n] with P(c) (P is monotone)
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (P(mid)) hi = mid;
      else lo = mid + 1;
    }
    i = lo;
  }
  if (i >= n) {
    u += 1;
    i = 0;
  }
}

// kind and kind-local index of tile i: bf16 sub-tile b (returns false) or 2-bit window k (true)
__device__ __forceinline__ bool tile_kind(const Lay& y, int i, int& local) {
  const int qb = q_before(y, i);
  if (q_before(y, i + 1) > qb) {
    local = qb;
    return true;
  }
  local = i - qb;
  return false;
}

// list entry {window, slot} of tile (u, i)
__device__ __forceinline__ int2 list_entry(const AttnParams& p, const Lay& y, int u, int i, int sub_tiles) {
  const State& st = p.st;
  const long long gu = (long long)p.layer * st.units + u;
  int loc;
  if (!tile_kind(y, i, loc)) return st.blist[gu * st.capb + loc / sub_tiles];
  return st.qlist[gu * st.capq + loc];
}

// descriptor of tile (u, i) from its list entry; false if it has no valid row (or is corrupt).
// d.i is the tile's index in the per-unit log-sum-exp array: bf16 sub-tiles first, then 2-bit.
// inew / opens: the tile of this step's appended token, and whether that token opens its window
// (then the other sub-tiles of the window, entry nbw - 1, are empty and their entry unread).
__device__ __forceinline__ bool describe(const AttnParams& p, const Lay& y, int u, int i, int2 ent, TileDesc& d,
                                         int inew, bool opens) {
  const State& st = p.st;
  const int W = st.geo.W;
  const int sub_tiles = W / 16;
  int loc;
  const bool is_q = tile_kind(y, i, loc);
  if (opens && !is_q && i != inew && loc / sub_tiles == y.nbw - 1) return false;
  d.u = u;
  d.i = is_q ? y.nbt + loc : loc;
  d.win = ent.x;
  d.slot = ent.y;
  if (!is_q) {
    d.kind = 0;
    d.sub = loc % sub_tiles;
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
      const int h = y.L - ent.x * W;
      hi = h < W ? h : W;
    }
    const int base = d.sub * 16;
    const int tl = lo - base, th = hi - base;
    d.lo = tl < 0 ? 0 : tl;
    d.hi = th > 16 ? 16 : th;
    return d.hi > d.lo;
  }
  d.kind = 1;
  d.sub = 0;
  if (ent.y < 0 || ent.y >= st.capq || ent.x < 0 || ent.x >= st.maxw) {
    atomicOr(st.err, ERR_TABLE);
    return false;
  }
  d.range = 0;   // the slot's range record: loaded by the caller (slot_range)
  d.lo = (ent.x == 0) ? st.n_sink : 0;
  d.hi = W;
  return true;
}

// a 2-bit tile's slot range record (qrange_word)
__device__ __forceinline__ int slot_range(const AttnParams& p, const TileDesc& d) {
  return p.st.qrange[((long long)p.layer * p.st.units + d.u) * p.st.capq + d.slot];
}

__device__ __forceinline__ const uint8_t* tile_src(const AttnParams& p, const TileDesc& d, unsigned& bytes) {
  const State& st = p.st;
  const long long gu = (long long)p.layer * st.units + d.u;
  if (d.kind == 0) {
    bytes = st.geo.sub_bytes();
    return st.bslab + ((gu * st.capb + d.slot) * (long long)st.geo.bslot_bytes()) + (long long)d.sub * st.geo.sub_bytes();
  }
  bytes = st.geo.qslot_bytes();
  return st.qslab + (gu * st.capq + d.slot) * (long long)st.geo.qslot_bytes();
}

// Index (in the interleaved tile order) of the bf16 sub-tile that holds the newest token,
// position L - 1: the sink tile, or the sub-tile of the last bf16 list entry (the current
// window has the highest index of the bf16 windows).  Identical for every unit of the layer.
__device__ __forceinline__ int newest_token_tile(const State& st, const Lay& y) {
  const int P = y.L - 1, W = st.geo.W;
  int loc = 0;   // bf16 tile number (bf16 list order)
  if (P >= st.n_sink) loc = (y.nbw - 1) * (W / 16) + (P - (P / W) * W) / 16;
  return bf16_tile_index(loc, y.ntiles, y.nbt);
}

// The decode step's own append, done at the start of the launch by the one warp that owns the
// tile holding the new token: open the token's window if the token starts it, then write K and
// V into the slot in fragment order.  The token's values are loaded together with the slot
// lookup (one round trip).  The stores are made visible at device scope and ordered, by the
// async-proxy fence, before the bulk copy that later reads the tile.  Returns the slot, -1 on
// error.
__device__ __forceinline__ int append_newest(const AttnParams& p, const Lay& y, int u, int lane) {
  const State& st = p.st;
  const Geo& g = st.geo;
  const int W = g.W, D = g.D;
  const long long gu = (long long)p.layer * st.units + u;
  const int P = y.L - 1, j = P / W;
  constexpr int MAXPAIRS = 2;   // channel pairs per lane (D <= 128)
  unsigned kk[MAXPAIRS];
  uint16_t v0[MAXPAIRS], v1[MAXPAIRS];
  const uint16_t* k = p.knew + (size_t)u * D;
  const uint16_t* v = p.vnew + (size_t)u * D;
#pragma unroll
  for (int i = 0; i < MAXPAIRS; ++i) {
    const int c = 2 * lane + 64 * i;
    if (c < D) {
      kk[i] = *reinterpret_cast<const unsigned*>(k + c);
      v0[i] = v[c];
      v1[i] = v[c + 1];
    }
  }
  int slot = -1;
  if (lane == 0) {
    if (P >= st.max_context || j >= st.maxw) {
      atomicOr(st.err, ERR_CAPACITY);
    } else {
      if (P % W == 0) slot = open_window(st, gu, j, y.nbw - 1);
      else slot = st.bslot[gu * st.maxw + j];
      if (P < st.n_sink && slot >= 0) slot = 0;
      if (slot < 0 || slot >= st.capb || (slot == 0 && P >= st.n_sink)) {
        atomicOr(st.err, ERR_TABLE);
        slot = -1;
      }
    }
  }
  slot = __shfl_sync(0xffffffffu, slot, 0);
  if (slot >= 0) {
    const int row = P < st.n_sink ? P : P - j * W;
    uint8_t* base = st.bslab + (gu * st.capb + slot) * (long long)g.bslot_bytes();
#pragma unroll
    for (int i = 0; i < MAXPAIRS; ++i) {
      const int c = 2 * lane + 64 * i;
      if (c < D) {
        *reinterpret_cast<unsigned*>(base + bf16_k_off(g, row, c)) = kk[i];
        *reinterpret_cast<uint16_t*>(base + bf16_v_off(g, row, c)) = v0[i];
        *reinterpret_cast<uint16_t*>(base + bf16_v_off(g, row, c + 1)) = v1[i];
      }
    }
    __threadfence();
    asm volatile("fence.proxy.async;" ::: "memory");
  }
  __syncwarp();
  return slot;
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
  static constexpr int OFF_KMIN = KCODE;
  static constexpr int OFF_KSCALE = KCODE + 4 * D;
  static constexpr int OFF_VCODE = KCODE + 8 * D;
  static constexpr int OFF_VMIN = OFF_VCODE + KCODE;
  static constexpr int OFF_VSCALE = OFF_VCODE + KCODE + 4 * W;
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

// N floats starting at p (16-byte vectors where possible)
template <int N>
__device__ __forceinline__ void load_floats(const float* p, float (&v)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const float4 f = reinterpret_cast<const float4*>(p)[i];
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
  } else {
    const float2 f = *reinterpret_cast<const float2*>(p);
    v[0] = f.x; v[1] = f.y;
  }
}

// Running softmax state of one warp for the unit it is working on.  Column n of every
// mma fragment is head n/2, "hi" part (n even) or "lo" remainder (n odd), so lane (g, t) owns
// head t: its accumulator pair (2t, 2t+1) holds that head's hi and lo parts for rows g, g+8.
// Scores are kept in the log2 domain against a reference maximum mref that is only raised when
// a tile's maximum exceeds it by more than 8 (so p <= 2^8): most tiles skip the rescale.
template <int MC>
struct RunState {
  float mref;      // head t
  float l;
  float zs;        // sum of p * z_V over 2-bit tokens (value offsets), partial over this lane's rows
  float O[MC][4];  // O^T fragments: rows = channels, columns 2t (hi) and 2t+1 (lo) of head t
};

// acc[mt][f][.] are split accumulators of the Q K^T products of token tile mt (summed here).
template <int MT, int NF, int MC, bool INT2, bool WIDE = false>
__device__ __forceinline__ void softmax_tile(float (&acc)[MT][NF][4], bool full, int lo, int hi, float bias,
                                             const float (&vz)[2 * MT], const float (&vs)[2 * MT], float scale_log2,
                                             RunState<MC>& st, unsigned (&Bp)[MT][2], float* lse_out, int G, int lane,
                                             bool pbf16 = false) {
  const int g = lane >> 2, t = lane & 3;
  float x[MT][2];   // rows g and g + 8 of each token tile
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = 0.f;
#pragma unroll
      for (int f = 0; f < NF; ++f) v += acc[mt][f][2 * j] + acc[mt][f][2 * j + 1];
      x[mt][j] = (v + bias) * scale_log2;
    }
  if (!full) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int row = mt * 16 + g + 8 * j;
        if (row < lo || row >= hi) x[mt][j] = -INFINITY;
      }
  }
  float mx = -INFINITY;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) mx = fmaxf(mx, fmaxf(x[mt][0], x[mt][1]));
  // only a lane that may exceed 2^8 needs the exact maximum of its head
  if (__any_sync(0xffffffffu, mx > st.mref + 8.f)) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(st.mref, mx);
    const float alpha = (st.mref == -INFINITY) ? 0.f : ex2(st.mref - mn);
    st.mref = mn;
    st.l *= alpha;
    st.zs *= alpha;
#pragma unroll
    for (int mc = 0; mc < MC; ++mc)
#pragma unroll
      for (int r = 0; r < 4; ++r) st.O[mc][r] *= alpha;
  }
  const float muse = st.mref == -INFINITY ? 0.f : st.mref;
  float pr[MT][2];
  float mass = 0.f, zadd = 0.f;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float pv = ex2(x[mt][j] - muse);
      pr[mt][j] = pv;
      mass += pv;
      if constexpr (INT2) zadd = fmaf(pv, vz[mt * 2 + j], zadd);
    }
  if constexpr (INT2) st.zs += zadd;
  mass += __shfl_xor_sync(0xffffffffu, mass, 4);
  mass += __shfl_xor_sync(0xffffffffu, mass, 8);
  mass += __shfl_xor_sync(0xffffffffu, mass, 16);
  st.l += mass;
  if (g == 0 && t < G) lse_out[t] = mass > 0.f ? muse + lg2(mass) : -INFINITY;
  // P^T fragments in D layout: (row g: hi, lo of head t), (row g+8: ...), then transposed
  // 2-bit values meet f16 codes (f16 truncated + remainder), or bf16 codes on a wide tile (WIDE,
  // or at run time pbf16)
  constexpr bool F16 = INT2 && !WIDE;
  const unsigned KEEP = (F16 && !pbf16) ? 0xFFFFE000u : 0xFFFF0000u;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    unsigned rr[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float y = pr[mt][j];
      if constexpr (INT2) y *= vs[mt * 2 + j];
      const float yh = __uint_as_float(__float_as_uint(y) & KEEP);
      if constexpr (F16) rr[j] = pbf16 ? pack_bf16x2_rz(yh, y - yh) : pack_f16x2_rz(yh, y - yh);
      else rr[j] = pack_bf16x2_rz(yh, y - yh);
    }
    Bp[mt][0] = movmatrix_t(rr[0]);
    Bp[mt][1] = movmatrix_t(rr[1]);
  }
}

// Keys stored pre-RoPE (QEvict reading notes, §4.4: quantized before the rotation, rotated again
// at their original positions): cos / sin of the angle (16 b + r) theta_i by angle addition from
// the block table (b) and the row-offset table (r).
__device__ __forceinline__ float2 rope_cs(float2 b, float2 o) {
  return make_float2(fmaf(b.x, o.x, -b.y * o.y), fmaf(b.y, o.x, b.x * o.y));
}
// The channel pair (x0, x1) rotated by (cos, sin), each rotated value as a tf32 truncated part
// and a tf32-truncated remainder (22 bits together; tf32 keeps float32's exponent range, so no
// key magnitude leaves it, and the bf16 query is exact in tf32).  In the m16n8k8 tf32 mma a lane
// holds k = t and k = t + 4 of its rows: k = t carries channel 2i and k = t + 4 channel 2i + 1 of
// the lane's pair i, the same mapping for the query's B fragment (b0 = q_2i, b1 = q_2i+1).
__device__ __forceinline__ void rope_rot_tf32(float x0, float x1, float2 cs, unsigned& h0, unsigned& h1, unsigned& l0,
                                              unsigned& l1) {
  const float y0 = fmaf(x0, cs.x, -x1 * cs.y);
  const float y1 = fmaf(x0, cs.y, x1 * cs.x);
  h0 = __float_as_uint(y0) & 0xFFFFE000u;
  h1 = __float_as_uint(y1) & 0xFFFFE000u;
  l0 = __float_as_uint(y0 - __uint_as_float(h0)) & 0xFFFFE000u;
  l1 = __float_as_uint(y1 - __uint_as_float(h1)) & 0xFFFFE000u;
}
constexpr int ROPE_OFF_STRIDE_PAD = 4;   // float2 padding of a row of the offset table in shared memory

template <int D, int W, bool ROPE = false>
__global__ void __launch_bounds__(ATTN_WARPS * 32, 1) qe_decode_attn_kernel(const AttnParams p) {
  using S = Shape<D, W>;
  constexpr int KS = S::KS, MC = S::MC, MT = S::MT, KT = S::KT, WPL = S::WPL, CW = S::CW, NST = S::NST;
  constexpr int SUBT = W / 16;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) unsigned long long bars[ATTN_WARPS][NST];
  __shared__ StageDesc descs[ATTN_WARPS][NST];
  __shared__ BatchDesc batches[ATTN_WARPS][BATCH];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = p.st.G;
  const int wg = blockIdx.x * ATTN_WARPS + warp;
  // The launch is a programmatic dependent of the kernel before it on the stream (the previous
  // layer's combine, which reads the split-K scratch this launch rewrites): the CTAs may be
  // resident early, but nothing is read or written before that kernel has completed.
  griddep_wait();
  // the layer's step-dependent counts live in shared memory (read when a batch of tiles is
  // described), not in registers the tile loop needs
  __shared__ Lay s_lay;
  if (threadIdx.x == 0) s_lay = make_lay(p.st, p.layer, p.pend, p.cb, p.cq, gridDim.x * ATTN_WARPS);
  constexpr int ROS = D / 2 + ROPE_OFF_STRIDE_PAD;
  __shared__ float2 s_roff[ROPE ? 16 * ROS : 1];
  if constexpr (ROPE) {
    for (int i = threadIdx.x; i < 16 * (D / 2); i += blockDim.x) s_roff[(i / (D / 2)) * ROS + i % (D / 2)] = p.rope_off[i];
  }
  // the combine launch may start as CTAs of this one leave (it waits for this grid's completion)
  griddep_launch_dependents();
  __syncthreads();
  const Lay& y = s_lay;
  // this warp's cost range [x_lo, x_hi) (lanes 0 and 1 compute the two ends at once), its units
  // u_first .. u_last, and r_lo, where the range starts inside unit u_first
  const RangeEnd e = range_end(y.Cu, y.NW, p.st.units, wg + (lane & 1));
  RangeEnd e_lo, e_hi;
  e_lo.x = __shfl_sync(0xffffffffu, e.x, 0);
  e_lo.c = __shfl_sync(0xffffffffu, e.c, 0);
  e_lo.k = __shfl_sync(0xffffffffu, e.k, 0);
  e_hi.x = __shfl_sync(0xffffffffu, e.x, 1);
  e_hi.c = __shfl_sync(0xffffffffu, e.c, 1);
  e_hi.k = __shfl_sync(0xffffffffu, e.k, 1);
  const long long x_lo = e_lo.x, x_hi = e_hi.x;
  const int u_first = e_lo.k + (e_lo.c >= y.Cu ? 1 : 0);
  const long long r_lo = e_lo.c >= y.Cu ? e_lo.c - y.Cu : e_lo.c;
  // the warps whose ranges meet unit u are u NW / units .. ; partial slot = warp - first warp
  auto slot_of = [&](int u) -> long long {
    return (long long)u * p.pslots + (wg - (int)udiv_fit((unsigned long long)u * (unsigned)y.NW, (unsigned)p.st.units));
  };
  if (x_lo >= x_hi) {   // empty range: leave an empty partial in the unit it falls into
    const int u = u_first;
    if (u < p.st.units && lane < G) p.part_ml[slot_of(u) * G + lane] = make_float2(-INFINITY, 0.f);
    return;
  }
  const int u_last = e_hi.k - (e_hi.c == 0 ? 1 : 0);
  // This decode step's appended token sits in tile inew of every unit; the warp that owns that
  // tile writes it first.  When the token opens its window, only that warp may use the window's
  // list entry (it writes it): the window's other sub-tiles are empty (rows past the token) and
  // describe() drops them without a look at the entry.
  const int inew = p.pend > 0 ? newest_token_tile(p.st, y) : -1;
  const bool opens = p.pend > 0 && (y.L - 1) % p.st.geo.W == 0;
  if (inew >= 0) {
    for (int u = u_first; u <= u_last; ++u) {
      const long long x = tile_start(p, y, u, inew);
      if (x >= x_lo && x < x_hi) append_newest(p, y, u, lane);
    }
  }

  uint8_t* stage_base = smem + (size_t)warp * NST * S::STAGE;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
    mbar_fence_init();
  }
  __syncwarp();

  // ---- producer: the warp describes BATCH tiles at a time (one per lane, empty tiles
  //      compacted out), then issues them one by one from shared memory; the first batch's
  //      lanes issue the range's first NST copies themselves
  BatchDesc* batch = batches[warp];
  int cu, ci;                        // cursor: first tile not yet described
  first_tile(p, y, u_first, r_lo, lane, cu, ci);
  bool range_done = !(cu < p.st.units && tile_start(p, y, cu, ci) < x_hi);
  int bcount = 0, bnext = 0;
  // pro: copies the batch issues itself (the prologue's first batch: NST, later batches: 0)
  auto describe_batch = [&](int pro) {
    while (!range_done) {
      int u = cu, i = ci + lane;
      while (i >= y.ntiles) { i -= y.ntiles; ++u; }
      const bool inr = u < p.st.units && tile_start(p, y, u, i) < x_hi;
      TileDesc d;
      bool ok = false;
      if (inr) ok = describe(p, y, u, i, list_entry(p, y, u, i, SUBT), d, inew, opens);
      const unsigned vb = __ballot_sync(0xffffffffu, ok);
      const int pos = __popc(vb & ((1u << lane) - 1));
      unsigned bytes = 0;
      const uint8_t* src = ok ? tile_src(p, d, bytes) : nullptr;
      // prologue: the lanes holding the first tiles issue their copies before the 2-bit tiles'
      // range records (a second dependent load) arrive
      if (ok && pos < pro) {
        const unsigned bar = smem_u32(&bars[warp][pos]);
        mbar_expect_tx(bar, bytes);
        bulk_g2s_hint(smem_u32(stage_base + (size_t)pos * S::STAGE), src, bytes, bar, l2_evict_first_policy());
      }
      if (ok && d.kind) d.range = slot_range(p, d);
      if (ok) {
        BatchDesc bd;
        bd.src = src;
        bd.bytes = bytes;
        bd.sd.u = u;
        bd.sd.lse_off = (u * y.ntiles + d.i) * G;
        bd.sd.meta = d.lo | (d.hi << 8) | (d.kind << 16);
        // 16-token block of the tile's first row (its position / 16; the sink tile is block 0)
        // (the default kernel: a 2-bit window's range record instead)
        // (keys stored pre-RoPE: the block, and bit 30 set when a 2-bit window's value products
        // need bf16 operands; the default kernel: a 2-bit window's range record)
        bd.sd.pad = ROPE ? (d.win < 0 ? 0 : d.win * (W / 16) + (d.kind == 0 ? d.sub : 0)) |
                               (d.kind && qrange_values_wide(d.range) ? (1 << 30) : 0)
                         : (d.kind ? d.range : 0);
        bd.pad = 0;
        batch[pos] = bd;
      }
      range_done = __any_sync(0xffffffffu, !inr);
      ci += BATCH;
      while (ci >= y.ntiles) { ci -= y.ntiles; ++cu; }
      bcount = __popc(vb);
      bnext = 0;
      __syncwarp();
      if (bcount > 0) {
        if (pro > 0) {   // stage descriptors of the copies issued above
          bnext = bcount < pro ? bcount : pro;
          if (lane < bnext) descs[warp][lane] = batch[lane].sd;
          __syncwarp();
        }
        return;
      }
    }
  };
  auto issue_next = [&](int stage) -> bool {
    if (bnext == bcount) {
      if (range_done) return false;
      describe_batch(0);
      if (bcount == 0) return false;
    }
    if (lane == 0) {
      const BatchDesc bd = batch[bnext];
      descs[warp][stage] = bd.sd;
      const unsigned bar = smem_u32(&bars[warp][stage]);
      mbar_expect_tx(bar, bd.bytes);
      // the tiles are read once per step: evict-first in L2
      bulk_g2s_hint(smem_u32(stage_base + (size_t)stage * S::STAGE), bd.src, bd.bytes, bar, l2_evict_first_policy());
    }
    ++bnext;
    return true;
  };
  describe_batch(NST);   // issues the copies of the range's first tiles
  int issued = bnext;
  for (int s = issued; s < NST; ++s) {
    if (!issue_next(s)) break;
    ++issued;
  }
  __syncwarp();

  // ---- consumer
  RunState<MC> rs;
  unsigned long long qf[KS][2];   // q of head g/2 at channels (16ks + 2t, +1), (+8, +9), as fp32 pairs
  unsigned qb[KS][2];      // bf16 B fragments: q of head g/2 in even columns, 0 in odd ones
  // keys stored pre-RoPE: tf32 B fragments of the two m16n8k8 per channel step (q_2i, q_2i+1 of
  // pair t, then of pair t + 4), q of head g/2 in even columns, 0 in odd ones
  unsigned qt[ROPE ? KS : 1][4];
  int qexp = 0;            // largest biased exponent of the unit's queries (qrange_wide)
  int cur_u = u_first;
  int q_unit = -1;
  auto reset = [&]() {
    rs.mref = -INFINITY;
    rs.l = 0.f;
    rs.zs = 0.f;
#pragma unroll
    for (int mc = 0; mc < MC; ++mc)
#pragma unroll
      for (int r = 0; r < 4; ++r) rs.O[mc][r] = 0.f;
  };
  auto flush = [&](int u) {
    const long long pidx = slot_of(u);
    float z = rs.zs;
    z += __shfl_xor_sync(0xffffffffu, z, 4);
    z += __shfl_xor_sync(0xffffffffu, z, 8);
    z += __shfl_xor_sync(0xffffffffu, z, 16);
    if (t < G) {
      float* po = p.part_o + (pidx * G + t) * D;
#pragma unroll
      for (int mc = 0; mc < MC; ++mc) {
        po[mc * 16 + g] = rs.O[mc][0] + rs.O[mc][1] + z;
        po[mc * 16 + g + 8] = rs.O[mc][2] + rs.O[mc][3] + z;
      }
      if (g == 0) p.part_ml[pidx * G + t] = make_float2(rs.mref, rs.l);
    }
  };
  reset();

  const int hh = g >> 1;               // head of the B columns this lane supplies
  const bool lo_col = (g & 1) != 0;    // ... and whether it is the remainder column
  // a waiting warp is suspended on the barrier (up to ~20 us per test) instead of spinning
  auto wait_tile = [&](int k) -> bool {
    const unsigned bar = smem_u32(&bars[warp][k % NST]);
    const unsigned parity = (k / NST) & 1;
    bool ok = true;
    if (!mbar_try_wait_sleep(bar, parity, 20000u)) {
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait_sleep(bar, parity, 20000u))
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
          ok = false;
          break;
        }
    }
    return __all_sync(0xffffffffu, ok);
  };
  bool timed_out = false;
  int k = 0;
  for (; k < issued; ++k) {
    const int s = k % NST;
    // (a test can make the k-th wait report expiry; the tile's copy has landed by then)
    if (!wait_tile(k) || k + 1 == p.debug_expire) { timed_out = true; break; }
    const StageDesc sd = descs[warp][s];
    const int d_lo = sd.meta & 0xFF, d_hi = (sd.meta >> 8) & 0xFF, d_kind = sd.meta >> 16;
    const uint8_t* sp = stage_base + (size_t)s * S::STAGE;
    while (sd.u > cur_u) {
      flush(cur_u);
      reset();
      ++cur_u;
    }
    if (q_unit != cur_u) {
      q_unit = cur_u;
      const int b = cur_u / p.st.Hkv, kvh = cur_u - b * p.st.Hkv;
      const uint16_t* qh = p.q + ((size_t)b * p.st.Hq + kvh * G + hh) * D;
      const bool act = hh < G;
      unsigned qmaxbits = 0u;   // largest |q| bits (bf16 pairs: both halves' magnitudes)
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const unsigned a0 = act ? *reinterpret_cast<const unsigned*>(qh + ks * 16 + 2 * t) : 0u;
        const unsigned a1 = act ? *reinterpret_cast<const unsigned*>(qh + ks * 16 + 8 + 2 * t) : 0u;
        qmaxbits = max(qmaxbits, max(max(a0 & 0x7FFFu, (a0 >> 16) & 0x7FFFu), max(a1 & 0x7FFFu, (a1 >> 16) & 0x7FFFu)));
        qf[ks][0] = f2_pack(bf16lo_to_f32(a0), bf16hi_to_f32(a0));
        qf[ks][1] = f2_pack(bf16lo_to_f32(a1), bf16hi_to_f32(a1));
        qb[ks][0] = lo_col ? 0u : a0;
        qb[ks][1] = lo_col ? 0u : a1;
        if constexpr (ROPE) {
          qt[ks][0] = lo_col ? 0u : (a0 << 16);
          qt[ks][1] = lo_col ? 0u : (a0 & 0xFFFF0000u);
          qt[ks][2] = lo_col ? 0u : (a1 << 16);
          qt[ks][3] = lo_col ? 0u : (a1 & 0xFFFF0000u);
        }
      }
      qexp = (int)(__reduce_max_sync(0xffffffffu, qmaxbits) >> 7);
    }
    float* lse_out = p.lse + sd.lse_off;
    if (d_kind == 0) {
      // ---- bf16 sub-tile: 16 tokens; independent accumulators shorten the mma dependency
      //      chains (two for stored keys, one per part for rotated keys)
      float acc[1][2][4] = {};
      if constexpr (ROPE) {
        // registers: (row g, pair 8 ks + t), (row g + 8, same), (row g, pair 8 ks + 4 + t), (row g + 8, same);
        // rotated keys meet the query as tf32 truncated + remainder parts, one m16n8k8 per pair
        // block of four pairs and part
        const float2* bt = p.rope_blk + (size_t)(sd.pad & 0x3FFFFFFF) * (D / 2);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint4 a = lds128(sp + ks * 512 + lane * 16);
          const int i0 = 8 * ks + t, i1 = i0 + 4;
          const float2 b0 = bt[i0], b1 = bt[i1];
          unsigned h[8], l[8];   // [pair block][row][channel of the pair]
          rope_rot_tf32(bf16lo_to_f32(a.x), bf16hi_to_f32(a.x), rope_cs(b0, s_roff[g * ROS + i0]), h[0], h[2], l[0], l[2]);
          rope_rot_tf32(bf16lo_to_f32(a.y), bf16hi_to_f32(a.y), rope_cs(b0, s_roff[(g + 8) * ROS + i0]), h[1], h[3], l[1],
                        l[3]);
          rope_rot_tf32(bf16lo_to_f32(a.z), bf16hi_to_f32(a.z), rope_cs(b1, s_roff[g * ROS + i1]), h[4], h[6], l[4], l[6]);
          rope_rot_tf32(bf16lo_to_f32(a.w), bf16hi_to_f32(a.w), rope_cs(b1, s_roff[(g + 8) * ROS + i1]), h[5], h[7], l[5],
                        l[7]);
          mma_tf32(acc[0][0], h[0], h[1], h[2], h[3], qt[ks][0], qt[ks][1]);
          mma_tf32(acc[0][1], l[0], l[1], l[2], l[3], qt[ks][0], qt[ks][1]);
          mma_tf32(acc[0][0], h[4], h[5], h[6], h[7], qt[ks][2], qt[ks][3]);
          mma_tf32(acc[0][1], l[4], l[5], l[6], l[7], qt[ks][2], qt[ks][3]);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint4 a = lds128(sp + ks * 512 + lane * 16);
          mma_bf16(acc[0][ks & 1], a.x, a.y, a.z, a.w, qb[ks][0], qb[ks][1]);
        }
      }
      const float vnone[2] = {0.f, 0.f};
      unsigned Bp[1][2];
      softmax_tile<1, 2, MC, false>(acc, d_lo == 0 && d_hi == 16, d_lo, d_hi, 0.f, vnone, vnone, p.scale_log2, rs,
                                    Bp, lse_out, G, lane);
#pragma unroll
      for (int mc = 0; mc < MC; ++mc) {
        const uint4 a = lds128(sp + 32 * D + mc * 512 + lane * 16);
        mma_bf16(rs.O[mc], a.x, a.y, a.z, a.w, Bp[0][0], Bp[0][1]);
      }
    } else {
      if constexpr (ROPE) {
        // ---- 2-bit window, keys stored pre-RoPE: W tokens
        const float* kmin = reinterpret_cast<const float*>(sp + S::OFF_KMIN);
        const float* kscale = reinterpret_cast<const float*>(sp + S::OFF_KSCALE);
        float vz[2 * MT], vs[2 * MT];
        load_floats<2 * MT>(reinterpret_cast<const float*>(sp + S::OFF_VMIN) + g * 2 * MT, vz);
        load_floats<2 * MT>(reinterpret_cast<const float*>(sp + S::OFF_VSCALE) + g * 2 * MT, vs);
        // codes arrive as 1 + code / 4: B = 4 p s_V, and the offset p . (z_V - 4 s_V) per token
#pragma unroll
        for (int i = 0; i < 2 * MT; ++i) {
          vs[i] *= 4.f;
          vz[i] -= vs[i];
        }
        float acc[MT][2][4] = {};
          // keys dequantized per element (one float32 fma), rotated at their positions, then split
          // into tf32 truncated + remainder parts against the tf32 query; register r of fragment
          // F holds the codes of channels 2i, 2i + 1 at bits 8 (F & 1) + 2 r and 16 above
          unsigned wk[WPL];
          load_words<WPL, CW>(sp, lane, wk);
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const ulonglong2 sc = *reinterpret_cast<const ulonglong2*>(kscale + ks * 16 + t * 4);
            const ulonglong2 zc = *reinterpret_cast<const ulonglong2*>(kmin + ks * 16 + t * 4);
            const float ksv[4] = {f2_lo(sc.x), f2_hi(sc.x), f2_lo(sc.y), f2_hi(sc.y)};
            const float kzv[4] = {f2_lo(zc.x), f2_hi(zc.x), f2_lo(zc.y), f2_hi(zc.y)};
            const int i0 = 8 * ks + t, i1 = i0 + 4;
            const float2 o[4] = {s_roff[g * ROS + i0], s_roff[(g + 8) * ROS + i0], s_roff[g * ROS + i1],
                                 s_roff[(g + 8) * ROS + i1]};
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              const int F = mt * KS + ks;
              const unsigned w = wk[F >> 1];
              const float2* bt = p.rope_blk + (size_t)((sd.pad & 0x3FFFFFFF) + mt) * (D / 2);
              const float2 b0 = bt[i0], b1 = bt[i1];
              unsigned h[8], l[8];   // [pair block][row][channel of the pair]
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                const int sh = 8 * (F & 1) + 2 * r;
                const int pc = (r >> 1) * 2;   // channel pair (2t, 2t+1) or (2t+8, 2t+9)
                const float x0 = fmaf((float)((w >> sh) & 3u), ksv[pc], kzv[pc]);
                const float x1 = fmaf((float)((w >> (sh + 16)) & 3u), ksv[pc + 1], kzv[pc + 1]);
                const int e = 4 * (r >> 1) + (r & 1);   // register r: row g + 8 (r & 1), pair block r >> 1
                rope_rot_tf32(x0, x1, rope_cs(r < 2 ? b0 : b1, o[r]), h[e], h[e + 2], l[e], l[e + 2]);
              }
              mma_tf32(acc[mt][0], h[0], h[1], h[2], h[3], qt[ks][0], qt[ks][1]);
              mma_tf32(acc[mt][1], l[0], l[1], l[2], l[3], qt[ks][0], qt[ks][1]);
              mma_tf32(acc[mt][0], h[4], h[5], h[6], h[7], qt[ks][2], qt[ks][3]);
              mma_tf32(acc[mt][1], l[4], l[5], l[6], l[7], qt[ks][2], qt[ks][3]);
            }
          }
        // values meet f16 codes (4 p s_V as f16 truncated + remainder, 22 bits), or bf16 codes
        // when the window's value scales could leave the f16 range (bit 30 of the descriptor)
        unsigned Bp[MT][2];
        const bool vwide = (sd.pad >> 30) & 1;
        softmax_tile<MT, 2, MC, true, false>(acc, d_lo == 0, d_lo, d_hi, 0.f, vz, vs, p.scale_log2, rs, Bp, lse_out,
                                             G, lane, vwide);
        // P V over the unpacked value codes (A = V^T: fragment F = mc KT + kt); token steps in
        // the outer loop, so consecutive mma go to the MC independent accumulators
        {
          unsigned wv[WPL];
          load_words<WPL, CW>(sp + S::OFF_VCODE, lane, wv);
          if (!vwide) {
#pragma unroll
            for (int kt = 0; kt < KT; ++kt)
#pragma unroll
              for (int mc = 0; mc < MC; ++mc) {
                const int F = mc * KT + kt;
                unsigned a[4];
                if (F & 1) unpack_half<1>(wv[F >> 1], a);
                else unpack_half<0>(wv[F >> 1], a);
                mma_f16(rs.O[mc], a[0], a[1], a[2], a[3], Bp[kt][0], Bp[kt][1]);
              }
          } else {
#pragma unroll
            for (int kt = 0; kt < KT; ++kt)
#pragma unroll
              for (int mc = 0; mc < MC; ++mc) {
                const int F = mc * KT + kt;
                unsigned a[4];
                if (F & 1) unpack_half_bf16<1>(wv[F >> 1], a);
                else unpack_half_bf16<0>(wv[F >> 1], a);
                mma_bf16(rs.O[mc], a[0], a[1], a[2], a[3], Bp[kt][0], Bp[kt][1]);
              }
          }
        }
      } else {
        if (!qrange_wide(sd.pad, qexp)) {
          // ---- 2-bit window: W tokens
          const float* kmin = reinterpret_cast<const float*>(sp + S::OFF_KMIN);
          const float* kscale = reinterpret_cast<const float*>(sp + S::OFF_KSCALE);
          // B fragments q s_K in f16: trunc part in even columns, remainder in odd ones.  The codes
          // arrive as 1 + code / 4, so logit / 4 = q s_K . A + q . (z_K - 4 s_K) / 4: the bias
          // accumulates q . (z_K - 4 s_K), the logit scale below carries the factor 4.
          unsigned qp[KS][2];
          unsigned long long bp2 = 0ull;
          const unsigned long long neg4 = f2_pack(-4.f, -4.f);
          const unsigned keep = lo_col ? 0xFFFFE000u : 0u;
  #pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const ulonglong2 sc = *reinterpret_cast<const ulonglong2*>(kscale + ks * 16 + t * 4);
            const ulonglong2 zc = *reinterpret_cast<const ulonglong2*>(kmin + ks * 16 + t * 4);
            bp2 = f2_fma(qf[ks][0], zc.x, bp2);
            bp2 = f2_fma(qf[ks][1], zc.y, bp2);
            const unsigned long long y01 = f2_mul(qf[ks][0], sc.x), y23 = f2_mul(qf[ks][1], sc.y);
            bp2 = f2_fma(y01, neg4, bp2);   // q . (z_K - 4 s_K)
            bp2 = f2_fma(y23, neg4, bp2);
            const unsigned long long k2 = ((unsigned long long)keep << 32) | keep;
            const unsigned long long r01 = f2_sub(y01, y01 & k2), r23 = f2_sub(y23, y23 & k2);
            qp[ks][0] = pack_f16x2_rz(f2_lo(r01), f2_hi(r01));
            qp[ks][1] = pack_f16x2_rz(f2_lo(r23), f2_hi(r23));
          }
          float bpart = 0.25f * (f2_lo(bp2) + f2_hi(bp2));
          bpart += __shfl_xor_sync(0xffffffffu, bpart, 1);
          bpart += __shfl_xor_sync(0xffffffffu, bpart, 2);
          const float bias = __shfl_sync(0xffffffffu, bpart, 8 * t);   // q . (z_K / 4 - s_K) of head t
          float vz[2 * MT], vs[2 * MT];
          load_floats<2 * MT>(reinterpret_cast<const float*>(sp + S::OFF_VMIN) + g * 2 * MT, vz);
          load_floats<2 * MT>(reinterpret_cast<const float*>(sp + S::OFF_VSCALE) + g * 2 * MT, vs);
          // codes arrive as 1 + code / 4: B = 4 p s_V, and the offset p . (z_V - 4 s_V) per token
  #pragma unroll
          for (int i = 0; i < 2 * MT; ++i) {
            vs[i] *= 4.f;
            vz[i] -= vs[i];
          }
          // Q K^T over the unpacked key codes (fragment F = mt KS + ks is half F % 2 of word F / 2);
          // channel-step parity splits the accumulators, and consecutive mma go to different
          // accumulators (2 MT independent chains)
          float acc[MT][2][4] = {};
          {
            unsigned wk[WPL];
            load_words<WPL, CW>(sp, lane, wk);
  #pragma unroll
            for (int ks = 0; ks < KS; ++ks)
  #pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                const int F = mt * KS + ks;
                unsigned a[4];
                if (F & 1) unpack_half<1>(wk[F >> 1], a);
                else unpack_half<0>(wk[F >> 1], a);
                mma_f16(acc[mt][ks & 1], a[0], a[1], a[2], a[3], qp[ks][0], qp[ks][1]);
              }
          }
          unsigned Bp[MT][2];
          softmax_tile<MT, 2, MC, true>(acc, d_lo == 0, d_lo, d_hi, bias, vz, vs, 4.f * p.scale_log2, rs, Bp, lse_out,
                                        G, lane);
          // P V over the unpacked value codes (A = V^T: fragment F = mc KT + kt); token steps in
          // the outer loop, so consecutive mma go to the MC independent accumulators
          {
            unsigned wv[WPL];
            load_words<WPL, CW>(sp + S::OFF_VCODE, lane, wv);
  #pragma unroll
            for (int kt = 0; kt < KT; ++kt)
  #pragma unroll
              for (int mc = 0; mc < MC; ++mc) {
                const int F = mc * KT + kt;
                unsigned a[4];
                if (F & 1) unpack_half<1>(wv[F >> 1], a);
                else unpack_half<0>(wv[F >> 1], a);
                mma_f16(rs.O[mc], a[0], a[1], a[2], a[3], Bp[kt][0], Bp[kt][1]);
              }
          }
        } else {
          // ---- 2-bit window whose products could leave the f16 range (qrange_wide): the same
          //      algebra on bf16 operands.  Keys: B = q s_K as three bf16 parts (truncated, the
          //      truncated remainder, the rest), exact together, in two mma passes into the same
          //      accumulators (pass one: parts one and two in the even and odd columns, pass two:
          //      part three in the even ones).  Values: B = 4 p s_V as bf16 truncated + remainder.
          const float* kmin = reinterpret_cast<const float*>(sp + S::OFF_KMIN);
          const float* kscale = reinterpret_cast<const float*>(sp + S::OFF_KSCALE);
          // the B operands of one channel step at a time, next to their mma (few live registers)
          float acc[MT][2][4] = {};
          unsigned long long bp2 = 0ull;
          const unsigned long long neg4 = f2_pack(-4.f, -4.f);
          {
            unsigned wk[WPL];
            load_words<WPL, CW>(sp, lane, wk);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              const ulonglong2 sc = *reinterpret_cast<const ulonglong2*>(kscale + ks * 16 + t * 4);
              const ulonglong2 zc = *reinterpret_cast<const ulonglong2*>(kmin + ks * 16 + t * 4);
              bp2 = f2_fma(qf[ks][0], zc.x, bp2);
              bp2 = f2_fma(qf[ks][1], zc.y, bp2);
              const unsigned long long y01 = f2_mul(qf[ks][0], sc.x), y23 = f2_mul(qf[ks][1], sc.y);
              bp2 = f2_fma(y01, neg4, bp2);
              bp2 = f2_fma(y23, neg4, bp2);
              const float y[4] = {f2_lo(y01), f2_hi(y01), f2_lo(y23), f2_hi(y23)};
              float pa[4], pb[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float h = __uint_as_float(__float_as_uint(y[i]) & 0xFFFF0000u);
                const float r = y[i] - h;
                const float m = __uint_as_float(__float_as_uint(r) & 0xFFFF0000u);
                pa[i] = lo_col ? m : h;
                pb[i] = lo_col ? 0.f : r - m;
              }
              const unsigned qa0 = pack_bf16x2_rz(pa[0], pa[1]), qa1 = pack_bf16x2_rz(pa[2], pa[3]);
              const unsigned qz0 = pack_bf16x2_rz(pb[0], pb[1]), qz1 = pack_bf16x2_rz(pb[2], pb[3]);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                const int F = mt * KS + ks;
                unsigned a[4];
                if (F & 1) unpack_half_bf16<1>(wk[F >> 1], a);
                else unpack_half_bf16<0>(wk[F >> 1], a);
                mma_bf16(acc[mt][ks & 1], a[0], a[1], a[2], a[3], qa0, qa1);
                mma_bf16(acc[mt][ks & 1], a[0], a[1], a[2], a[3], qz0, qz1);
              }
            }
          }
          float bpart = 0.25f * (f2_lo(bp2) + f2_hi(bp2));
          bpart += __shfl_xor_sync(0xffffffffu, bpart, 1);
          bpart += __shfl_xor_sync(0xffffffffu, bpart, 2);
          const float bias = __shfl_sync(0xffffffffu, bpart, 8 * t);
          float vz[2 * MT], vs[2 * MT];
          load_floats<2 * MT>(reinterpret_cast<const float*>(sp + S::OFF_VMIN) + g * 2 * MT, vz);
          load_floats<2 * MT>(reinterpret_cast<const float*>(sp + S::OFF_VSCALE) + g * 2 * MT, vs);
#pragma unroll
          for (int i = 0; i < 2 * MT; ++i) {
            vs[i] *= 4.f;
            vz[i] -= vs[i];
          }
          unsigned Bp[MT][2];
          softmax_tile<MT, 2, MC, true, true>(acc, d_lo == 0, d_lo, d_hi, bias, vz, vs, 4.f * p.scale_log2, rs, Bp,
                                              lse_out, G, lane);
          {
            unsigned wv[WPL];
            load_words<WPL, CW>(sp + S::OFF_VCODE, lane, wv);
  #pragma unroll
            for (int kt = 0; kt < KT; ++kt)
  #pragma unroll
              for (int mc = 0; mc < MC; ++mc) {
                const int F = mc * KT + kt;
                unsigned a[4];
                if (F & 1) unpack_half_bf16<1>(wv[F >> 1], a);
                else unpack_half_bf16<0>(wv[F >> 1], a);
                mma_bf16(rs.O[mc], a[0], a[1], a[2], a[3], Bp[kt][0], Bp[kt][1]);
              }
          }
        }
      }
    }
    __syncwarp();
    if (issue_next(s)) ++issued;   // refill this stage
    __syncwarp();
  }
  if (timed_out) {
    // report, then give the copies still in flight (the expired tile's included) a bounded
    // chance to land before exiting
    if (lane == 0) atomicOr(p.st.err, ERR_TIMEOUT);
    for (int kk = k; kk < issued; ++kk) wait_tile(kk);
    return;
  }
  while (cur_u <= u_last) {
    flush(cur_u);
    reset();
    ++cur_u;
  }
}

// ------------------------------------------------------------------------------ combine
// One CTA per unit (COMBINE_THREADS = 4 x 128 threads).  Thread (h, c) = (tid / D, tid % D)
// merges the partials of query head h < G at channel c and writes o_h = sum / l; every thread
// also takes list entries (bf16 windows, then 2-bit ones), turns their tiles' log2-sum-exps into
// mass, sums it over the G heads and adds it to the window's float32 score (eq. (1) with the GQA
// group sum).  Warps 0..G-1 compute each head's global statistics.  The partial slots follow
// from the attention launch's warp ranges.
//
// The combine is launched as a programmatic dependent of the attention launch: its CTAs start
// as attention CTAs leave, compute the layer's counts from the header (the attention read the
// same header and does not change it), load what the attention does not write (list entries
// and scores of windows that existed before this step), then wait for the attention grid
// (griddepcontrol.wait: completion and memory flush) and issue every load of partials and
// tile log-sum-exps at once.  The last CTA to finish commits the new length.
constexpr int COMBINE_THREADS = 512;
constexpr int MAXP = COMBINE_MAXP;
constexpr int COMBINE_PR = 32;     // partials per thread held in registers (more are re-read)
constexpr int COMBINE_EPT = 2;     // list entries per thread per round
constexpr int COMBINE_MAXSUB = 4;  // 16-token sub-tiles per bf16 window (w <= 64)

// partial slots of unit u: one per warp whose position range meets [u Cu, (u+1) Cu)
__device__ __forceinline__ int unit_partials(const CombineParams& p, const Lay& y, int u) {
  const long long w0 = (long long)u * p.NW / p.st.units;
  const long long w1 = (((long long)u + 1) * y.Cu - 1) * p.NW / y.C;
  int np = (int)(w1 - w0 + 1);
  if (np > p.pslots) np = p.pslots;
  return np;
}

// head h's global max over the partials, the scale of each partial and log2 of the normaliser;
// executed by one warp
__device__ __forceinline__ void head_stats(const CombineParams& p, int u, int np, int h, float* s_sc, float& inv,
                                           float& lse) {
  const int lane = threadIdx.x & 31;
  const int G = p.st.G;
  const float2* ml0 = p.part_ml + (size_t)u * p.pslots * G + h;
  float2 ml[MAXP / 32];
#pragma unroll
  for (int j = 0; j < MAXP / 32; ++j) {
    const int k = lane + 32 * j;
    ml[j] = k < np ? ml0[(size_t)k * G] : make_float2(-INFINITY, 0.f);
  }
  float M = -INFINITY;
#pragma unroll
  for (int j = 0; j < MAXP / 32; ++j) M = fmaxf(M, ml[j].x);
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float Ls = 0.f;
#pragma unroll
  for (int j = 0; j < MAXP / 32; ++j) {
    const int k = lane + 32 * j;
    const float sc = ml[j].y > 0.f ? ex2(ml[j].x - Mu) : 0.f;
    if (k < np) s_sc[k] = sc;
    Ls = fmaf(ml[j].y, sc, Ls);
  }
  for (int o = 16; o; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
  inv = 1.f / Ls;
  lse = Mu + lg2(Ls);
}

template <int D>
__global__ void __launch_bounds__(COMBINE_THREADS) qe_attn_combine_kernel(const CombineParams p) {
  const int u = blockIdx.x;
  const int G = p.st.G;
  const long long gu = (long long)p.layer * p.st.units + u;
  __shared__ float s_sc[4][MAXP];
  __shared__ float s_inv[4], s_lse[4];
  const int tid = threadIdx.x, warp = tid >> 5;
  const Lay y = make_lay(p.st, p.layer, p.pend, p.cb, p.cq, p.NW);   // counts incl. the pending token
  const int np = unit_partials(p, y, u);
  const int W = p.st.geo.W, sub_tiles = W / 16;
  const int nent = y.nbw + y.nq;
  const bool opens = p.pend > 0 && (y.L - 1) % W == 0;
  constexpr int EPT = COMBINE_EPT, MAXSUB = COMBINE_MAXSUB;
  auto load_ent = [&](int e) -> int2 {
    if (e < y.nbw) return p.st.blist[gu * p.st.capb + e];
    if (e < nent) return p.st.qlist[gu * p.st.capq + (e - y.nbw)];
    return make_int2(-1, -1);
  };
  // first round of this thread's entries and their scores (before the wait)
  int2 ent[EPT];
  float sc[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int e = tid + j * COMBINE_THREADS;
    const bool late = opens && e == y.nbw - 1;
    ent[j] = (e < nent && !late) ? load_ent(e) : make_int2(-1, -1);
    sc[j] = (ent[j].x >= 0 && ent[j].x < p.st.maxw) ? p.st.score[gu * p.st.maxw + ent[j].x] : 0.f;
  }
  griddep_wait();
  // the next layer's attention may now take the SMs this grid leaves (it waits for completion)
  griddep_launch_dependents();
  // ---- loads of this thread's partial outputs (head h, channel c) and tile log-sum-exps
  const int h = tid / D, c = tid - h * D;
  const bool out_thread = h < G;
  const float* po = p.part_o + ((size_t)u * p.pslots * G + h) * D + c;
  float v[COMBINE_PR];
#pragma unroll
  for (int k = 0; k < COMBINE_PR; ++k) v[k] = (out_thread && k < np) ? po[(size_t)k * G * D] : 0.f;
  auto load_lse = [&](int e, const int2 en, float (&ls)[MAXSUB][4]) {
#pragma unroll
    for (int s2 = 0; s2 < MAXSUB; ++s2)
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) ls[s2][hh] = -INFINITY;
    if (e >= nent || en.x < 0) return;
    if (e < y.nbw) {
      const int lo = (en.x == 0) ? p.st.n_sink : 0;
      int hi = y.L - en.x * W;
      hi = hi < W ? hi : W;
#pragma unroll
      for (int s2 = 0; s2 < MAXSUB; ++s2) {
        if (s2 >= sub_tiles) break;
        const int tl = lo - 16 * s2, th = hi - 16 * s2;
        if ((th > 16 ? 16 : th) <= (tl < 0 ? 0 : tl)) continue;
        const float* lp = p.lse + ((size_t)u * y.ntiles + e * sub_tiles + s2) * G;
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
          if (hh < G) ls[s2][hh] = lp[hh];
      }
    } else {
      const float* lp = p.lse + ((size_t)u * y.ntiles + y.nbt + (e - y.nbw)) * G;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh)
        if (hh < G) ls[0][hh] = lp[hh];
    }
  };
  if (opens) {   // the window this step opened: its entry now, its score is 0
#pragma unroll
    for (int j = 0; j < EPT; ++j)
      if (tid + j * COMBINE_THREADS == y.nbw - 1) {
        ent[j] = load_ent(y.nbw - 1);
        sc[j] = 0.f;
      }
  }
  float ls[EPT][MAXSUB][4];
#pragma unroll
  for (int j = 0; j < EPT; ++j) load_lse(tid + j * COMBINE_THREADS, ent[j], ls[j]);
  // ---- head statistics
  if (warp < G) {
    float inv, lse;
    head_stats(p, u, np, warp, s_sc[warp], inv, lse);
    if ((tid & 31) == 0) {
      s_inv[warp] = inv;
      s_lse[warp] = lse;
    }
  }
  __syncthreads();
  // ---- outputs
  if (out_thread) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < COMBINE_PR; ++k)
      if (k < np && s_sc[h][k] != 0.f) acc = fmaf(v[k], s_sc[h][k], acc);
    for (int k = COMBINE_PR; k < np; ++k)
      if (s_sc[h][k] != 0.f) acc = fmaf(po[(size_t)k * G * D], s_sc[h][k], acc);
    const float o = acc * s_inv[h];
    const int bb = u / p.st.Hkv, kvh = u - bb * p.st.Hkv;
    const size_t oi = ((size_t)bb * p.st.Hq + kvh * G + h) * D + c;
    if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = o;
    else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
  }
  // ---- scores
  for (int r0 = 0; r0 < nent; r0 += COMBINE_THREADS * EPT) {
    if (r0 > 0) {   // later rounds (a unit with more entries than one round holds)
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const int e = r0 + tid + j * COMBINE_THREADS;
        ent[j] = e < nent ? load_ent(e) : make_int2(-1, -1);
        sc[j] = (ent[j].x >= 0 && ent[j].x < p.st.maxw) ? p.st.score[gu * p.st.maxw + ent[j].x] : 0.f;
        if (opens && e == y.nbw - 1) sc[j] = 0.f;
        load_lse(e, ent[j], ls[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = r0 + tid + j * COMBINE_THREADS;
      if (e >= nent || ent[j].x < 0) continue;
      if (ent[j].x >= p.st.maxw) {
        atomicOr(p.st.err, ERR_TABLE);
        continue;
      }
      float dS = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < MAXSUB; ++s2)
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
          if (hh < G) dS += ex2(ls[j][s2][hh] - s_lse[hh]);
      if (p.delta) p.delta[(long long)u * p.st.maxw + ent[j].x] = dS;
      else p.st.score[gu * p.st.maxw + ent[j].x] = sc[j] + dS;
    }
  }
  // The last CTA to finish commits the new length: every CTA read the header when it started,
  // before its count.
  __syncthreads();
  if (tid == 0) {
    LayerDev* hd = p.st.ldev + p.layer;
    if (atomicAdd(&hd->done, 1u) == gridDim.x - 1) {
      hd->L = y.L;
      hd->done = 0;
    }
  }
}

// ------------------------------------------------------------------------------ launchers
template <int D, int W>
static size_t attn_smem_bytes() {
  using S = Shape<D, W>;
  return (size_t)ATTN_WARPS * S::NST * S::STAGE;
}

template <int D, int W>
static cudaError_t launch_attn_t(const AttnParams& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(ATTN_WARPS * 32);
  cfg.dynamicSmemBytes = attn_smem_bytes<D, W>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.rope_blk) return cudaLaunchKernelEx(&cfg, qe_decode_attn_kernel<D, W, true>, p);
  return cudaLaunchKernelEx(&cfg, qe_decode_attn_kernel<D, W, false>, p);
}

template <int D, int W>
static cudaError_t prepare_attn_t() {
  cudaError_t e = cudaFuncSetAttribute(qe_decode_attn_kernel<D, W, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)attn_smem_bytes<D, W>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(qe_decode_attn_kernel<D, W, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_smem_bytes<D, W>());
}

// kernel attributes, set once (outside any stream capture)
cudaError_t prepare_attn_kernels(int D, int W) {
  if (D == 128 && W == 32) return prepare_attn_t<128, 32>();
  if (D == 128 && W == 16) return prepare_attn_t<128, 16>();
  if (D == 128 && W == 64) return prepare_attn_t<128, 64>();
  if (D == 64 && W == 16) return prepare_attn_t<64, 16>();
  if (D == 64 && W == 32) return prepare_attn_t<64, 32>();
  if (D == 64 && W == 64) return prepare_attn_t<64, 64>();
  return cudaErrorInvalidValue;
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

// programmatic dependent of the attention launch before it on the stream (see the kernel)
cudaError_t launch_attn_combine(const CombineParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.st.units);
  cfg.blockDim = dim3(COMBINE_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.st.geo.D == 128) return cudaLaunchKernelEx(&cfg, qe_attn_combine_kernel<128>, p);
  return cudaLaunchKernelEx(&cfg, qe_attn_combine_kernel<64>, p);
}

int attn_warps_per_cta() { return ATTN_WARPS; }

// A launch with the attention launch's shape (grid, block, dynamic shared memory, programmatic
// serialization) that does nothing: timing it between two events gives the part of an event
// time that is launch and event overhead rather than the kernel's work.
__global__ void __launch_bounds__(ATTN_WARPS * 32, 1) qe_empty_attn_shaped_kernel(int* never) {
  extern __shared__ unsigned char smem_unused[];
  if (never != nullptr && threadIdx.x == 0 && blockIdx.x == 0x7fffffff) never[0] = smem_unused[0];
}

cudaError_t time_empty_attn_launch(int D, int W, int grid, int n, cudaStream_t stream, double* us) {
  size_t smem = 0;
  if (D == 128 && W == 32) smem = attn_smem_bytes<128, 32>();
  else if (D == 128 && W == 16) smem = attn_smem_bytes<128, 16>();
  else if (D == 128 && W == 64) smem = attn_smem_bytes<128, 64>();
  else if (D == 64 && W == 16) smem = attn_smem_bytes<64, 16>();
  else if (D == 64 && W == 32) smem = attn_smem_bytes<64, 32>();
  else if (D == 64 && W == 64) smem = attn_smem_bytes<64, 64>();
  else return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(qe_empty_attn_shaped_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  // all launches enqueued back to back, each between its own two events, as the timed attention
  // launches are; one synchronization at the end
  std::vector<cudaEvent_t> ev(2 * (size_t)n, nullptr);
  for (size_t i = 0; i < ev.size() && e == cudaSuccess; ++i) e = cudaEventCreate(&ev[i]);
  for (int i = 0; i < n && e == cudaSuccess; ++i) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(ATTN_WARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaEventRecord(ev[2 * i], stream);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, qe_empty_attn_shaped_kernel, (int*)nullptr);
    if (e == cudaSuccess) e = cudaEventRecord(ev[2 * i + 1], stream);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  double total = 0;
  for (int i = 0; i < n && e == cudaSuccess; ++i) {
    float t = 0;
    e = cudaEventElapsedTime(&t, ev[2 * i], ev[2 * i + 1]);
    total += t;
  }
  for (cudaEvent_t x : ev)
    if (x) cudaEventDestroy(x);
  if (e == cudaSuccess && us) *us = n > 0 ? 1000.0 * total / n : 0.0;
  return e;
}

// Persistent grid: one CTA per SM, but few enough warps that a unit meets at most pslots - 2
// warp ranges.
int attn_grid(int n_sm, int units, int pslots) {
  long long g = ((long long)(pslots - 2) * units) / ATTN_WARPS;
  if (g > n_sm) g = n_sm;
  return g < 1 ? 1 : (int)g;
}

}  // namespace qe
