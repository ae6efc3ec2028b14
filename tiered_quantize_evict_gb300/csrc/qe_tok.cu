// qe_tok.cu -- kernels of the five-tier per-token cache (HqeKV reading notes §3.1-§3.5; layout in
// qe_tok.cuh): the single-token append, the split-K decode attention over BF16 / 4-bit / 2-bit /
// 1-bit tiles with per-token logits for the importance, the split merge with the score update,
// and the demote-only re-rank that rebuilds the pools.
//
// Attention (what it computes): for each unit and its G query heads, o_h = softmax(q_h K^T /
// sqrt(d)) V over the kept tokens, every quantized token dequantized as x = code * s + z (uniform,
// eq. (2)) or x = c_code * s + m (normal, eq. (4) centers +-Phi^-1(3/4)); on the steps that
// count towards the importance, each token's attention mass summed over the G heads is added to
// its float32 score.
//
// GB300 design:
//  * persistent grid of 12-warp CTAs; the layer's units x tiles sequence is cut into one
//    cost-weighted range per warp (stream-K over per-unit costs that differ after re-ranking); a
//    warp streams its range through a private two-stage ring filled by cp.async.bulk;
//  * Q K^T and P V run on the tensor cores (mma.m16n8k16, fp32 accumulate): b-bit codes are
//    turned into the operands 1 + code / 2^b with one shift and one and-or per register (bf16 for
//    keys, which meet the bf16 queries exactly; f16 for values, which meet P split into a
//    truncated and a remainder column); the per-token key scale and offset are applied to the
//    logits, the value scale goes into P and the value offset into a running sum;
//  * the per-token importance leaves the attention as log2-domain logits; the merge kernel
//    turns them into probability mass once the unit's normaliser is known.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qe_exact_stats.cuh"
#include "qe_tok.cuh"
#include "qe_tok_kernels.h"

namespace qe {

constexpr int TK_WARPS = 12;
constexpr int TK_STAGE_TOTAL = 196608;
constexpr unsigned long long TK_WAIT_NS = 200000000ull;   // 0.2 s
constexpr float TK_NQ1_C = 0.67448975f;                   // Phi^-1(3/4) rounded to float32
constexpr int TK_MERGE_THREADS = 512;
constexpr int TK_MERGE_SPLIT = 4;       // CTAs per unit: each takes a quarter of the outputs and tokens
constexpr int TK_RERANK_THREADS = 256;

// ------------------------------------------------------------------------------ unit geometry
struct TkUnit {
  int t[5];            // tiles per segment (pools BF16, INT4, INT2, 1-bit, then the tail)
  int n[5];            // tokens per segment
  long long s0[6];     // cost offset of each segment; s0[5] = the unit's cost
  int tok0[5];         // token-slot offset of each segment (16 x tiles before it)
};

__device__ __forceinline__ TkUnit tk_unit(const TokState& s, int layer, int u, int n_tail) {
  const int4 c = *reinterpret_cast<const int4*>(s.cnt + ((long long)layer * s.units + u) * 4);
  TkUnit g;
  g.n[0] = c.x; g.n[1] = c.y; g.n[2] = c.z; g.n[3] = c.w; g.n[4] = n_tail;
  long long x = 0;
  int tk = 0;
#pragma unroll
  for (int z = 0; z < 5; ++z) {
    g.t[z] = (g.n[z] + 15) >> 4;
    g.s0[z] = x;
    g.tok0[z] = tk;
    x += (long long)g.t[z] * s.cost[z];
    tk += 16 * g.t[z];
  }
  g.s0[5] = x;
  return g;
}

// cost offset of unit u: ranked prefix plus u tails
__device__ __forceinline__ long long tk_X(const long long* cum, int u, long long tail_cost) {
  return cum[u] + (long long)u * tail_cost;
}

// The units holding cost positions xa and xb, found together by the warp: each round the lanes
// test 32 units spread over each remaining interval (one load each, all in flight at once)
// instead of a binary search's chain of dependent loads.  X(lo) <= x holds throughout (X(0) = 0).
__device__ __forceinline__ int2 tk_units_of(const long long* cum, int units, long long tail_cost, long long xa,
                                            long long xb, int lane) {
  int lo0 = 0, hi0 = units - 1, lo1 = 0, hi1 = units - 1;
  while (hi0 > lo0 || hi1 > lo1) {
    const bool p0 = tk_X(cum, search32_unit(lo0, hi0, lane), tail_cost) <= xa;
    const bool p1 = tk_X(cum, search32_unit(lo1, hi1, lane), tail_cost) <= xb;
    const unsigned b0 = __ballot_sync(0xffffffffu, p0) | 1u, b1 = __ballot_sync(0xffffffffu, p1) | 1u;
    search32_narrow(lo0, hi0, 31 - __clz(b0));   // the last lane whose unit starts at or before x
    search32_narrow(lo1, hi1, 31 - __clz(b1));
  }
  return make_int2(lo0, lo1);
}

// a[i] for a runtime i, by unrolled selects: the small per-unit arrays stay in registers
template <typename T, int N>
__device__ __forceinline__ T tk_pick(const T (&a)[N], int i) {
  T r = a[0];
#pragma unroll
  for (int k = 1; k < N; ++k)
    if (i == k) r = a[k];
  return r;
}

__device__ __forceinline__ const uint8_t* tk_tile_src(const TokState& s, int layer, int buf, int u, int z, int k) {
  if (z == 4) return s.tail + (tk_tail_tok_index(s, layer, buf, u) / 16 + k) * (long long)s.g.bf_tile();
  return s.pool[z] + (tk_pool_tile_index(s, z, layer, buf, u) + k) * (long long)tk_tile_bytes(s, z);
}

// ------------------------------------------------------------------------------ helpers
__device__ __forceinline__ uint4 tk_lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

// one test of an mbarrier phase that may suspend the thread until the phase completes (at most
// about 20 us)
__device__ __forceinline__ bool tk_try_wait(unsigned bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return done != 0;
}

template <int WPL>
__device__ __forceinline__ void tk_load_words(const uint8_t* blk, int lane, unsigned (&w)[WPL]) {
  constexpr int CW = WPL < 4 ? WPL : 4;
#pragma unroll
  for (int c = 0; c < WPL / CW; ++c) {
    const uint8_t* src = blk + (c * 32 + lane) * (CW * 4);
    if constexpr (CW == 4) {
      const uint4 v = tk_lds128(src);
      w[c * 4 + 0] = v.x; w[c * 4 + 1] = v.y; w[c * 4 + 2] = v.z; w[c * 4 + 3] = v.w;
    } else if constexpr (CW == 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      w[c * 2 + 0] = v.x; w[c * 2 + 1] = v.y;
    } else {
      w[c] = *reinterpret_cast<const unsigned*>(src);
    }
  }
}

// register r of step k (inside a word) as the operand pair 1 + code / 2^B: bf16 (EB = 7 mantissa
// bits, ONE = 0x3F80) or f16 (EB = 10, ONE = 0x3C00)
template <int B, int EB, unsigned ONE>
__device__ __forceinline__ unsigned tk_pair(unsigned w, int k, int r) {
  const int sh = (EB - B) - B * (4 * k + r);
  const unsigned x = sh >= 0 ? (w << sh) : (w >> (-sh));
  constexpr unsigned MASK = (((1u << B) - 1u) << (EB - B)) * 0x00010001u;
  return (x & MASK) | (ONE * 0x00010001u);
}

template <int MC>
struct TkRun {
  float mref, l, zs;
  float O[MC][4];
};

// Online softmax of one 16-token tile (rows g, g + 8 of this lane, head t).  Q: per-row key
// scale and offset (logit = ks v + kb) and per-row value scale (into P) and offset (into zs).
// lg: this tile's per-token logits (row * G + head), or null.
template <int MC, bool Q>
__device__ __forceinline__ void tk_softmax(float (&acc)[2][4], int nvalid, const float (&ksc)[2], const float (&kbi)[2],
                                           const float (&vz)[2], const float (&vs)[2], float scale_log2, TkRun<MC>& st,
                                           unsigned (&Bp)[2], float* lg, int G, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float x[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float v = (acc[0][2 * j] + acc[0][2 * j + 1]) + (acc[1][2 * j] + acc[1][2 * j + 1]);
    x[j] = (Q ? fmaf(v, ksc[j], kbi[j]) : v) * scale_log2;
    if (g + 8 * j >= nvalid) x[j] = -INFINITY;
  }
  if (lg != nullptr && t < G) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (g + 8 * j < nvalid) lg[(g + 8 * j) * G + t] = x[j];
  }
  float mx = fmaxf(x[0], x[1]);
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
  float pr[2];
  float mass = 0.f, zadd = 0.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    pr[j] = ex2(x[j] - muse);
    mass += pr[j];
    if constexpr (Q) zadd = fmaf(pr[j], vz[j], zadd);
  }
  if constexpr (Q) st.zs += zadd;
  st.l += mass;   // this lane's rows only: the flush sums the partial normalisers of a head
  constexpr unsigned KEEP = Q ? 0xFFFFE000u : 0xFFFF0000u;
  unsigned rr[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float y = pr[j];
    if constexpr (Q) y *= vs[j];
    const float yh = __uint_as_float(__float_as_uint(y) & KEEP);
    rr[j] = Q ? pack_f16x2_rz(yh, y - yh) : pack_bf16x2_rz(yh, y - yh);
  }
  Bp[0] = movmatrix_t(rr[0]);
  Bp[1] = movmatrix_t(rr[1]);
}

// (z_eff, s_eff) with x = z_eff + s_eff code: uniform (min, scale) as stored; normal (mean, std)
// with centers -+c: (m - c s, 2 c s)
__device__ __forceinline__ float2 tk_affine(float2 p, bool normal) {
  if (!normal) return p;
  return make_float2(fmaf(-TK_NQ1_C, p.y, p.x), 2.f * TK_NQ1_C * p.y);
}

struct TkDesc {
  int u, kind;
  int ntile;       // tiles in this stage (consecutive tiles of one segment)
  int rem;         // tokens of the segment from the stage's first tile on
  int tokslot;     // token slot of the first tile
  int pad[3];
};

// Tiles one stage carries: a BF16 tile fills it; quantized tiles of a segment are staged
// together (up to 64 d bytes), so every stage moves about as many bytes.
template <int D>
__device__ __forceinline__ int tk_per_stage(int z) {
  if (z == 0 || z == 4) return 1;
  return (64 * D) / (4 * D * tk_bits(z) + 256);
}

struct TkAttnArgs {
  TokState st;
  int layer, pend;
  const uint16_t* knew;   // this step's appended token (K, V: [units][D]) to write first, or null
  const uint16_t* vnew;
  const uint16_t* q;
  float scale_log2;
  float* part_o;
  float2* part_ml;
  float* logits;
  int lg_cap;
  int debug_expire;   // qe_debug_inject: k >= 1 reports the k-th tile wait as expired after it landed
};

template <int D>
__device__ __forceinline__ void tk_tile_bf16(const uint8_t* sp, int nvalid, const unsigned (&qb)[D / 16][2],
                                             TkRun<D / 16>& rs, float* lg, float scale_log2, int G, int lane) {
  constexpr int KS = D / 16, MC = D / 16;
  float acc[2][4] = {};
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const uint4 a = tk_lds128(sp + ks * 512 + lane * 16);
    mma_bf16(acc[ks & 1], a.x, a.y, a.z, a.w, qb[ks][0], qb[ks][1]);
  }
  const float none[2] = {0.f, 0.f};
  unsigned Bp[2];
  tk_softmax<MC, false>(acc, nvalid, none, none, none, none, scale_log2, rs, Bp, lg, G, lane);
#pragma unroll
  for (int mc = 0; mc < MC; ++mc) {
    const uint4 a = tk_lds128(sp + 32 * D + mc * 512 + lane * 16);
    mma_bf16(rs.O[mc], a.x, a.y, a.z, a.w, Bp[0], Bp[1]);
  }
}

// 1-bit keys: the four registers of a channel step are built after one shift of the code word,
// register r as 1 + code 2^(r - 4) (its code at mantissa bit 3 + r).  The channels of registers
// 2 and 3 meet the query divided by 4 (qb1, exact), so a row's codes all weigh 2^-4 (row g) or
// 2^-3 (row g + 8); the row's key scale takes the factor back, and q1sum (the query summed with
// the same 1 / 4 on those channels) replaces qsum in the offset.
template <int D, int B>
__device__ __forceinline__ void tk_tile_q(const uint8_t* sp, int nvalid, bool normal, const unsigned (&qb)[D / 16][2],
                                          const unsigned (&qb1)[D / 16], float qsum, float q1sum, TkRun<D / 16>& rs,
                                          float* lg, float scale_log2, int G, int lane) {
  constexpr int KS = D / 16, MC = D / 16, WPL = D * B / 64, PW = 4 / B;
  constexpr float TWO_B = (float)(1 << B);
  const TokGeo geo{D};
  const int g = lane >> 2;
  // per-row parameters (rows g, g + 8)
  const float2* kp = reinterpret_cast<const float2*>(sp + geo.off_kpar(B));
  const float2* vp = reinterpret_cast<const float2*>(sp + geo.off_vpar(B));
  float ksc[2], kbi[2], vz[2], vs[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float2 ka = tk_affine(kp[g + 8 * j], normal);
    const float2 va = tk_affine(vp[g + 8 * j], normal);
    if constexpr (B == 1) {
      ksc[j] = (j ? 8.f : 16.f) * ka.y;
      kbi[j] = fmaf(-ksc[j], q1sum, ka.x * qsum);
    } else {
      ksc[j] = TWO_B * ka.y;
      kbi[j] = fmaf(-TWO_B, ka.y, ka.x) * qsum;
    }
    vs[j] = TWO_B * va.y;
    vz[j] = fmaf(-TWO_B, va.y, va.x);
  }
  float acc[2][4] = {};
  {
    unsigned wk[WPL];
    tk_load_words<WPL>(sp, lane, wk);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const unsigned w = wk[ks / PW];
      const int k = ks % PW;
      if constexpr (B == 1) {
        const int sh = 4 * k - 3;   // bit 4 k (register 0 of step k) to bit 3
        const unsigned x = sh >= 0 ? (w >> sh) : (w << (-sh));
        mma_bf16(acc[ks & 1], (x & 0x00080008u) | 0x3F803F80u, (x & 0x00100010u) | 0x3F803F80u,
                 (x & 0x00200020u) | 0x3F803F80u, (x & 0x00400040u) | 0x3F803F80u, qb[ks][0], qb1[ks]);
      } else {
        mma_bf16(acc[ks & 1], tk_pair<B, 7, 0x3F80u>(w, k, 0), tk_pair<B, 7, 0x3F80u>(w, k, 1),
                 tk_pair<B, 7, 0x3F80u>(w, k, 2), tk_pair<B, 7, 0x3F80u>(w, k, 3), qb[ks][0], qb[ks][1]);
      }
    }
  }
  unsigned Bp[2];
  tk_softmax<MC, true>(acc, nvalid, ksc, kbi, vz, vs, scale_log2, rs, Bp, lg, G, lane);
  {
    unsigned wv[WPL];
    tk_load_words<WPL>(sp + geo.off_vcode(B), lane, wv);
#pragma unroll
    for (int mc = 0; mc < MC; ++mc) {
      const unsigned w = wv[mc / PW];
      const int k = mc % PW;
      mma_f16(rs.O[mc], tk_pair<B, 10, 0x3C00u>(w, k, 0), tk_pair<B, 10, 0x3C00u>(w, k, 1),
              tk_pair<B, 10, 0x3C00u>(w, k, 2), tk_pair<B, 10, 0x3C00u>(w, k, 3), Bp[0], Bp[1]);
    }
  }
}

// The decode step's own append, by the one warp that owns the tail tile holding the new token:
// K and V into the tile in fragment order, its position and a zero score.  The stores are made
// visible at device scope and ordered, by the async-proxy fence, before the bulk copy that later
// reads the tile.
__device__ __forceinline__ void tk_append_newest(const TokState& s, int layer, int buf, int u, int idx, int pos,
                                                 const uint16_t* kn, const uint16_t* vn, int lane) {
  const int D = s.g.D;
  if (idx >= s.cap_tail) {
    if (lane == 0) atomicOr(s.err, ERR_CAPACITY);
    return;
  }
  const long long tb = tk_tail_tok_index(s, layer, buf, u);
  uint8_t* tile = s.tail + (tb / 16 + idx / 16) * (long long)s.g.bf_tile();
  const Geo g16{D, 16};
  const int row = idx & 15;
#pragma unroll
  for (int i = 0; i < 2; ++i) {   // channel pairs 2 lane + 64 i (D <= 128)
    const int c = 2 * lane + 64 * i;
    if (c < D) {
      const size_t src = (size_t)u * D + c;
      const unsigned kk = *reinterpret_cast<const unsigned*>(kn + src);
      const uint16_t v0 = vn[src], v1 = vn[src + 1];
      *reinterpret_cast<unsigned*>(tile + bf16_k_off(g16, row, c)) = kk;
      *reinterpret_cast<uint16_t*>(tile + bf16_v_off(g16, row, c)) = v0;
      *reinterpret_cast<uint16_t*>(tile + bf16_v_off(g16, row, c + 1)) = v1;
    }
  }
  if (lane == 0) {
    s.tail_pos[tb + idx] = pos;
    s.tail_score[tb + idx] = 0.f;
  }
  __threadfence();
  asm volatile("fence.proxy.async;" ::: "memory");
  __syncwarp();
}

// whether this decode step adds to the importance (the last score_window steps of a period)
__device__ __forceinline__ bool tk_scoring(const TokState& s, int step_before) {
  const int sidx = step_before + 1;
  return s.score_window == 0 || sidx > s.period - s.score_window;
}

template <int D>
__global__ void __launch_bounds__(TK_WARPS * 32, 1) tk_attn_kernel(const TkAttnArgs p) {
  constexpr int KS = D / 16, MC = D / 16;
  constexpr int STAGE = 64 * D;   // a BF16 tile, the largest
  constexpr int NST = TK_STAGE_TOTAL / (TK_WARPS * STAGE) < 4 ? TK_STAGE_TOTAL / (TK_WARPS * STAGE) : 4;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) unsigned long long bars[TK_WARPS][NST];
  __shared__ TkDesc descs[TK_WARPS][NST];
  const TokState& S = p.st;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = S.G;
  const int NW = gridDim.x * TK_WARPS;
  const int wg = blockIdx.x * TK_WARPS + warp;
  // The launch is a programmatic dependent of the kernel before it on the stream (the previous
  // layer's merge, which reads the split-K scratch this launch rewrites): nothing is read or
  // written before that kernel has completed.
  griddep_wait();
  const TokLayer hd = S.hdr[p.layer];
  const int n_tail = hd.n_tail + p.pend;
  const int buf = hd.buf;
  const bool scoring = tk_scoring(S, hd.step);
  griddep_launch_dependents();
  const long long* cum = S.cum + (long long)p.layer * (S.units + 1);
  const long long tail_cost = (long long)S.cost[4] * ((n_tail + 15) >> 4);
  const long long C = tk_X(cum, S.units, tail_cost);
  // this warp's cost range [x_lo, x_hi) (lanes 0 and 1 compute the two ends at once)
  const long long xe = ((long long)(wg + (lane & 1)) * C + NW - 1) / NW;
  const long long x_lo = __shfl_sync(0xffffffffu, xe, 0), x_hi = __shfl_sync(0xffffffffu, xe, 1);
  if (x_lo >= x_hi) {   // empty range: an empty partial in the unit it falls into
    if (x_lo < C) {
      const int u = tk_units_of(cum, S.units, tail_cost, x_lo, x_lo, lane).x;
      if (lane < G) p.part_ml[((long long)wg + u) * G + lane] = make_float2(-INFINITY, 0.f);
    }
    return;
  }
  const int2 uf = tk_units_of(cum, S.units, tail_cost, x_lo, x_hi - 1, lane);
  const int u_first = uf.x, u_last = uf.y;

  // this step's appended token (the last tail slot of every unit), written by the warp whose
  // range holds its tail tile, before that warp issues any copy
  if (p.knew) {
    const int idx = n_tail - 1, pc = tk_per_stage<D>(4), ts = (idx >> 4) / pc;   // the stage holding it
    for (int u = u_first; u <= u_last; ++u) {
      const TkUnit uu = tk_unit(S, p.layer, u, n_tail);
      const long long start = tk_X(cum, u, tail_cost) + uu.s0[4] + (long long)ts * pc * S.cost[4];
      if (start >= x_lo && start < x_hi) tk_append_newest(S, p.layer, buf, u, idx, hd.L, p.knew, p.vnew, lane);
    }
  }

  uint8_t* stage_base = smem + (size_t)warp * NST * STAGE;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(smem_u32(&bars[warp][s]), 1);
    mbar_fence_init();
  }
  __syncwarp();

  // ---- producer cursor (lane-uniform): unit cu, segment cz, tile ck
  int cu = u_first;
  TkUnit un = tk_unit(S, p.layer, cu, n_tail);
  long long ux = tk_X(cum, cu, tail_cost);
  int cz = 0, ck = 0;
  bool cvalid = true;
  // the cursor walks stages: stage k of segment z holds tiles [k pc, (k + 1) pc) (pc tiles per
  // stage) and starts at cost s0[z] + k pc cost[z]
  int cost[5];   // per-tile cost of each segment kind, in registers
#pragma unroll
  for (int z = 0; z < 5; ++z) cost[z] = S.cost[z];
  auto nstages = [&](int z) -> int { const int pc = tk_per_stage<D>(z); return (tk_pick(un.t, z) + pc - 1) / pc; };
  {
    // first stage whose start >= x_lo
    const long long r = x_lo - ux;
    cz = 5;
    for (int z = 0; z < 5; ++z) {
      if (un.t[z] == 0) continue;
      const long long step = (long long)tk_per_stage<D>(z) * cost[z];
      const long long last = un.s0[z] + (long long)(nstages(z) - 1) * step;
      if (r <= last) {
        cz = z;
        ck = r <= un.s0[z] ? 0 : (int)((r - un.s0[z] + step - 1) / step);
        break;
      }
    }
    if (cz == 5) {   // past the unit's last stage start: the next unit's first stage
      ++cu;
      if (cu >= S.units) cvalid = false;
      else {
        un = tk_unit(S, p.layer, cu, n_tail);
        ux = tk_X(cum, cu, tail_cost);
        cz = 0;
        ck = 0;
        while (cz < 5 && tk_pick(un.t, cz) == 0) ++cz;
      }
    }
  }
  auto advance = [&]() {
    ++ck;
    if (ck < nstages(cz)) return;
    ck = 0;
    ++cz;
    while (cz < 5 && tk_pick(un.t, cz) == 0) ++cz;
    if (cz < 5) return;
    ++cu;
    if (cu >= S.units) {
      cvalid = false;
      return;
    }
    un = tk_unit(S, p.layer, cu, n_tail);
    ux = tk_X(cum, cu, tail_cost);
    cz = 0;
    while (cz < 5 && tk_pick(un.t, cz) == 0) ++cz;
  };
  auto issue_next = [&](int stage) -> bool {
    if (!cvalid || cz >= 5) return false;
    const int pc = tk_per_stage<D>(cz);
    const long long start = ux + tk_pick(un.s0, cz) + (long long)ck * pc * tk_pick(cost, cz);
    if (start >= x_hi) return false;
    if (lane == 0) {
      const int kind = cz;
      const int t0 = ck * pc;
      const int tz = tk_pick(un.t, cz);
      const int nt = tz - t0 < pc ? tz - t0 : pc;
      const unsigned bytes = (unsigned)(nt * tk_tile_bytes(S, kind == 4 ? TK_TAIL : kind));
      TkDesc d;
      d.u = cu;
      d.kind = kind;
      d.ntile = nt;
      d.rem = tk_pick(un.n, cz) - 16 * t0;
      d.tokslot = tk_pick(un.tok0, cz) + 16 * t0;
      descs[warp][stage] = d;
      const unsigned bar = smem_u32(&bars[warp][stage]);
      mbar_expect_tx(bar, bytes);
      // the tiles are read once per step: evict-first in L2
      bulk_g2s_hint(smem_u32(stage_base + (size_t)stage * STAGE), tk_tile_src(S, p.layer, buf, cu, kind, t0), bytes, bar,
                    l2_evict_first_policy());
    }
    advance();
    return true;
  };
  int issued = 0;
  for (int s = 0; s < NST; ++s) {
    if (!issue_next(s)) break;
    ++issued;
  }
  __syncwarp();

  // ---- consumer
  TkRun<MC> rs;
  unsigned qb[KS][2];
  unsigned qb1[KS];   // qb[.][1] / 4, for 1-bit keys
  float qsum = 0.f, q1sum = 0.f;
  int cur_u = u_first, q_unit = -1;
  const int hh = g >> 1;
  const bool lo_col = (g & 1) != 0;
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
    const long long slot = (long long)wg + u;
    float z = rs.zs, l = rs.l;
    z += __shfl_xor_sync(0xffffffffu, z, 4);
    z += __shfl_xor_sync(0xffffffffu, z, 8);
    z += __shfl_xor_sync(0xffffffffu, z, 16);
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    if (t < G) {
      float* po = p.part_o + (slot * G + t) * D;
#pragma unroll
      for (int mc = 0; mc < MC; ++mc) {
        po[mc * 16 + g] = rs.O[mc][0] + rs.O[mc][1] + z;
        po[mc * 16 + g + 8] = rs.O[mc][2] + rs.O[mc][3] + z;
      }
      if (g == 0) p.part_ml[slot * G + t] = make_float2(rs.mref, l);
    }
  };
  reset();
  // a waiting warp is suspended on the barrier (up to ~20 us per test) instead of spinning
  auto wait_tile = [&](int k) -> bool {
    const unsigned bar = smem_u32(&bars[warp][k % NST]);
    const unsigned parity = (k / NST) & 1;
    bool ok = true;
    if (!tk_try_wait(bar, parity)) {
      const unsigned long long t0 = globaltimer_ns();
      while (!tk_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > TK_WAIT_NS) {
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
    if (!wait_tile(k) || k + 1 == p.debug_expire) { timed_out = true; break; }
    const TkDesc d = descs[warp][s];
    const uint8_t* sp = stage_base + (size_t)s * STAGE;
    while (d.u > cur_u) {
      flush(cur_u);
      reset();
      ++cur_u;
    }
    if (q_unit != cur_u) {
      q_unit = cur_u;
      const int b = cur_u / S.Hkv, kvh = cur_u - b * S.Hkv;
      const uint16_t* qh = p.q + ((size_t)b * S.Hq + kvh * G + hh) * D;
      const bool act = hh < G;
      float part = 0.f, part1 = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const unsigned a0 = act ? *reinterpret_cast<const unsigned*>(qh + ks * 16 + 2 * t) : 0u;
        const unsigned a1 = act ? *reinterpret_cast<const unsigned*>(qh + ks * 16 + 8 + 2 * t) : 0u;
        part += (bf16lo_to_f32(a0) + bf16hi_to_f32(a0)) + (bf16lo_to_f32(a1) + bf16hi_to_f32(a1));
        qb[ks][0] = lo_col ? 0u : a0;
        qb[ks][1] = lo_col ? 0u : a1;
        // q / 4 on channels 8..15 of the step, for 1-bit keys: exact while q / 4 stays a normal
        // float32 (|q| >= 2^-124); below that the bf16 truncation drops bits.  The offset sum
        // takes the truncated operands themselves, so it matches what the tensor core multiplies
        // in every case.
        const unsigned q4 = (__float_as_uint(0.25f * bf16lo_to_f32(a1)) >> 16) |
                            (__float_as_uint(0.25f * bf16hi_to_f32(a1)) & 0xFFFF0000u);
        part1 += (bf16lo_to_f32(a0) + bf16hi_to_f32(a0)) + (bf16lo_to_f32(q4) + bf16hi_to_f32(q4));
        qb1[ks] = lo_col ? 0u : q4;
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      part1 += __shfl_xor_sync(0xffffffffu, part1, 1);
      part1 += __shfl_xor_sync(0xffffffffu, part1, 2);
      qsum = __shfl_sync(0xffffffffu, part, 8 * t);     // sum of q over the channels, head t
      q1sum = __shfl_sync(0xffffffffu, part1, 8 * t);   // the same with q / 4 on channels 8..15 of each step
    }
    float* lg = scoring ? p.logits + ((long long)d.u * p.lg_cap + d.tokslot) * G : nullptr;
    const int nv0 = d.rem < 16 ? d.rem : 16;
    switch (d.kind) {
      case 0:
      case 4: tk_tile_bf16<D>(sp, nv0, qb, rs, lg, p.scale_log2, G, lane); break;
      case 1:
      case 2:
      case 3: {
        const int b = tk_bits(d.kind);
        const int tb = 4 * D * b + 256;
        for (int i = 0; i < d.ntile; ++i) {
          const int r = d.rem - 16 * i;
          const int nv = r < 16 ? r : 16;
          const uint8_t* ti = sp + i * tb;
          float* lgi = lg ? lg + 16 * i * G : nullptr;
          if (d.kind == 1) tk_tile_q<D, 4>(ti, nv, false, qb, qb1, qsum, q1sum, rs, lgi, p.scale_log2, G, lane);
          else if (d.kind == 2) tk_tile_q<D, 2>(ti, nv, false, qb, qb1, qsum, q1sum, rs, lgi, p.scale_log2, G, lane);
          else tk_tile_q<D, 1>(ti, nv, true, qb, qb1, qsum, q1sum, rs, lgi, p.scale_log2, G, lane);
        }
        break;
      }
      default: break;
    }
    __syncwarp();
    if (issue_next(s)) ++issued;
    __syncwarp();
  }
  if (timed_out) {
    if (lane == 0) atomicOr(S.err, ERR_TIMEOUT);
    for (int kk = k; kk < issued; ++kk) wait_tile(kk);   // copies in flight, the expired one's too
    return;
  }
  while (cur_u <= u_last) {
    flush(cur_u);
    reset();
    ++cur_u;
  }
}

// ------------------------------------------------------------------------------ append
// Single-token append: the token goes to the tail at index n_tail (its length is committed by
// the decode step's merge, or by tk_commit_kernel).
__global__ void tk_append1_kernel(TokState s, int layer, const uint16_t* __restrict__ k, const uint16_t* __restrict__ v) {
  const TokLayer hd = s.hdr[layer];
  const int D = s.g.D;
  const int u = blockIdx.x;
  const int c = 2 * threadIdx.x;
  if (c >= D) return;
  const int idx = hd.n_tail;
  if (idx >= s.cap_tail) {
    if (threadIdx.x == 0) atomicOr(s.err, ERR_CAPACITY);
    return;
  }
  const long long tb = tk_tail_tok_index(s, layer, hd.buf, u);
  uint8_t* tile = s.tail + (tb / 16 + idx / 16) * (long long)s.g.bf_tile();
  const Geo g16{D, 16};
  const int row = idx & 15;
  const size_t src = (size_t)u * D + c;
  *reinterpret_cast<unsigned*>(tile + bf16_k_off(g16, row, c)) = *reinterpret_cast<const unsigned*>(k + src);
  *reinterpret_cast<uint16_t*>(tile + bf16_v_off(g16, row, c)) = v[src];
  *reinterpret_cast<uint16_t*>(tile + bf16_v_off(g16, row, c + 1)) = v[src + 1];
  if (threadIdx.x == 0) {
    s.tail_pos[tb + idx] = hd.L;
    s.tail_score[tb + idx] = 0.f;
  }
}

// Multi-token append of n tokens at length L0 = hd.L.  prefill (L0 == 0): the sink and the last
// n_recent tokens go to the tail, the rest to the ranked BF16 pool; otherwise all to the tail.
__global__ void tk_append_kernel(TokState s, int layer, int n, int prefill, const uint16_t* __restrict__ k,
                                 const uint16_t* __restrict__ v) {
  const TokLayer hd = s.hdr[layer];
  const int D = s.g.D;
  const Geo g16{D, 16};
  const long long total = (long long)s.units * n * (D / 2);
  const int mid_lo = s.n_sink < n ? s.n_sink : n;
  int mid_hi = n - s.n_recent;
  if (mid_hi < mid_lo) mid_hi = mid_lo;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    const int c = 2 * (int)(e % (D / 2));
    const long long ti = e / (D / 2);
    const int i = (int)(ti % n);
    const int u = (int)(ti / n);
    uint8_t* tile;
    int row, idx;
    int* posp;
    float* scp;
    if (prefill && i >= mid_lo && i < mid_hi) {
      idx = i - mid_lo;
      if (idx >= s.cap[0]) { atomicOr(s.err, ERR_CAPACITY); continue; }
      const long long b0 = tk_pool_tok_index(s, 0, layer, hd.buf, u);
      tile = s.pool[0] + (tk_pool_tile_index(s, 0, layer, hd.buf, u) + idx / 16) * (long long)s.g.bf_tile();
      posp = s.pos[0] + b0 + idx;
      scp = s.score[0] + b0 + idx;
    } else {
      idx = prefill ? (i < mid_lo ? i : mid_lo + (i - mid_hi)) : hd.n_tail + i;
      if (idx >= s.cap_tail) { atomicOr(s.err, ERR_CAPACITY); continue; }
      const long long tb = tk_tail_tok_index(s, layer, hd.buf, u);
      tile = s.tail + (tb / 16 + idx / 16) * (long long)s.g.bf_tile();
      posp = s.tail_pos + tb + idx;
      scp = s.tail_score + tb + idx;
    }
    row = idx & 15;
    const size_t src = ((size_t)u * n + i) * D + c;
    *reinterpret_cast<unsigned*>(tile + bf16_k_off(g16, row, c)) = *reinterpret_cast<const unsigned*>(k + src);
    *reinterpret_cast<uint16_t*>(tile + bf16_v_off(g16, row, c)) = v[src];
    *reinterpret_cast<uint16_t*>(tile + bf16_v_off(g16, row, c + 1)) = v[src + 1];
    if (c == 0) {
      *posp = hd.L + i;
      *scp = 0.f;
    }
  }
}

// Header update after a multi-token append (one thread): length, tail count and, after a
// prefill, the ranked BF16 count of every unit and the cost prefix.
__global__ void tk_commit_kernel(TokState s, int layer, int n, int prefill) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  TokLayer& hd = s.hdr[layer];
  int* cnt = s.cnt + (long long)layer * s.units * 4;
  long long* cum = s.cum + (long long)layer * (s.units + 1);
  if (prefill) {
    const int mid_lo = s.n_sink < n ? s.n_sink : n;
    int mid_hi = n - s.n_recent;
    if (mid_hi < mid_lo) mid_hi = mid_lo;
    hd.n_tail = mid_lo + (n - mid_hi);
    const long long c0 = (long long)s.cost[0] * ((mid_hi - mid_lo + 15) >> 4);
    cum[0] = 0;
    for (int u = 0; u < s.units; ++u) {
      cnt[u * 4 + 0] = mid_hi - mid_lo;
      cnt[u * 4 + 1] = cnt[u * 4 + 2] = cnt[u * 4 + 3] = 0;
      cum[u + 1] = cum[u] + c0;
    }
  } else {
    hd.n_tail += n;
  }
  hd.L += n;
}

// ------------------------------------------------------------------------------ merge
struct TkMergeArgs {
  TokState st;
  int layer, pend, NW;
  const float* part_o;
  const float2* part_ml;
  const float* logits;
  int lg_cap;
  void* out;
  int out_fp32;
};

// TK_MERGE_SPLIT CTAs per unit: merge the partials of the warps whose ranges met the unit, write o_h, and on
// scoring steps add each token's mass (sum over the G heads of 2^(logit - lse_h)) to its score.
// A programmatic dependent of the attention launch.  The last CTA commits the appended token.
template <int D>
__global__ void __launch_bounds__(TK_MERGE_THREADS) tk_merge_kernel(const TkMergeArgs p) {
  extern __shared__ float s_sc[];   // [G][np]
  __shared__ float s_inv[4], s_lse[4];
  __shared__ bool s_last;
  const TokState& S = p.st;
  const int u = blockIdx.x / TK_MERGE_SPLIT, part = blockIdx.x - u * TK_MERGE_SPLIT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = S.G;
  const TokLayer hd = S.hdr[p.layer];
  const int n_tail = hd.n_tail + p.pend;
  const bool scoring = tk_scoring(S, hd.step);
  const long long* cum = S.cum + (long long)p.layer * (S.units + 1);
  const long long tail_cost = (long long)S.cost[4] * ((n_tail + 15) >> 4);
  const long long C = tk_X(cum, S.units, tail_cost);
  const long long X0 = tk_X(cum, u, tail_cost), X1 = tk_X(cum, u + 1, tail_cost);
  const long long w0 = X0 * p.NW / C, w1 = (X1 - 1) * p.NW / C;
  const int np = (int)(w1 - w0 + 1);
  const long long slot0 = w0 + u;
  const TkUnit un = tk_unit(S, p.layer, u, n_tail);
  griddep_wait();
  // the next layer's attention may now take the SMs this grid leaves (it waits for completion)
  griddep_launch_dependents();
  // Output element (h, c) of this CTA's share is summed by TPE adjacent threads, each over the
  // partials k = q, q + TPE, ...; their first loads are issued here, before the head
  // statistics that weight them.
  constexpr int TPE = 4, PF = 8;   // threads per element, partials per thread per round
  const int e_per = (G * D + TK_MERGE_SPLIT - 1) / TK_MERGE_SPLIT;   // <= TK_MERGE_THREADS / TPE
  const int e_end = (part + 1) * e_per < G * D ? (part + 1) * e_per : G * D;
  const int e = part * e_per + tid / TPE, q = tid % TPE;
  const bool has_e = tid / TPE < e_per && e < e_end;
  const int h_e = has_e ? e / D : 0, c_e = has_e ? e - h_e * D : 0;
  float pv[PF];
  auto load_round = [&](int k0) {
#pragma unroll
    for (int j = 0; j < PF; ++j) {
      const int k = k0 + q + TPE * j;
      pv[j] = (has_e && k < np) ? __ldg(p.part_o + ((slot0 + k) * G + h_e) * D + c_e) : 0.f;
    }
  };
  load_round(0);
  if (warp < G) {
    const int h = warp;
    float M = -INFINITY;
    for (int k = lane; k < np; k += 32) M = fmaxf(M, p.part_ml[(slot0 + k) * G + h].x);
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Mu = M == -INFINITY ? 0.f : M;
    float Ls = 0.f;
    for (int k = lane; k < np; k += 32) {
      const float2 ml = p.part_ml[(slot0 + k) * G + h];
      const float sc = ml.y > 0.f ? ex2(ml.x - Mu) : 0.f;
      s_sc[h * np + k] = sc;
      Ls = fmaf(ml.y, sc, Ls);
    }
    for (int o = 16; o; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane == 0) {
      s_inv[h] = 1.f / Ls;
      s_lse[h] = Mu + lg2(Ls);
    }
  }
  __syncthreads();
  {
    float acc = 0.f;
    for (int k0 = 0; k0 < np; k0 += TPE * PF) {
      if (k0 > 0) load_round(k0);
#pragma unroll
      for (int j = 0; j < PF; ++j) {
        const int k = k0 + q + TPE * j;
        if (has_e && k < np) {
          const float w = s_sc[h_e * np + k];
          if (w != 0.f) acc = fmaf(pv[j], w, acc);   // an empty partial (never written) weighs 0
        }
      }
    }
#pragma unroll
    for (int o = 1; o < TPE; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (has_e && q == 0) {
      const float o = acc * s_inv[h_e];
      const int bb = u / S.Hkv, kvh = u - bb * S.Hkv;
      const size_t oi = ((size_t)bb * S.Hq + kvh * G + h_e) * D + c_e;
      if (p.out_fp32) reinterpret_cast<float*>(p.out)[oi] = o;
      else reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
    }
  }
  if (scoring) {
    // The scored tokens of the pools and the tail (sink tokens are never scored) as one range,
    // split evenly over the unit's CTAs; NF tokens per thread in flight.
    const float* lgu = p.logits + (long long)u * p.lg_cap * G;
    int base[6];
    base[0] = 0;
#pragma unroll
    for (int z = 0; z < 5; ++z) {
      const int first = z < 4 ? 0 : S.n_sink;
      base[z + 1] = base[z] + (un.n[z] > first ? un.n[z] - first : 0);
    }
    const int per = (base[5] + TK_MERGE_SPLIT - 1) / TK_MERGE_SPLIT;
    const int lo = part * per;
    const int hi = lo + per < base[5] ? lo + per : base[5];
    constexpr int NF = 8;
    for (int i0 = lo + tid; i0 < hi; i0 += NF * TK_MERGE_THREADS) {
      float m[NF], old[NF];
      float* dst[NF];
#pragma unroll
      for (int j = 0; j < NF; ++j) {
        const int gi = i0 + j * TK_MERGE_THREADS;
        m[j] = 0.f;
        old[j] = 0.f;
        dst[j] = nullptr;
        if (gi < hi) {
          int z = 0;
          while (z < 4 && gi >= base[z + 1]) ++z;
          const int i = gi - base[z] + (z < 4 ? 0 : S.n_sink);
          dst[j] = (z < 4 ? S.score[z] + tk_pool_tok_index(S, z, p.layer, hd.buf, u)
                          : S.tail_score + tk_tail_tok_index(S, p.layer, hd.buf, u)) + i;
          const float* lg = lgu + (long long)(un.tok0[z] + i) * G;
          for (int h = 0; h < G; ++h) m[j] += ex2(__ldg(lg + h) - s_lse[h]);
          old[j] = *dst[j];
        }
      }
#pragma unroll
      for (int j = 0; j < NF; ++j)
        if (dst[j]) *dst[j] = old[j] + m[j];
    }
  }
  // commit: the last CTA advances the header
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(S.done + p.layer, 1u);
    s_last = prev == (unsigned)(S.units * TK_MERGE_SPLIT) - 1;
  }
  __syncthreads();
  if (s_last && tid == 0) {
    TokLayer& h = S.hdr[p.layer];
    h.L += p.pend;
    h.n_tail += p.pend;
    h.step += 1;
    S.done[p.layer] = 0;
  }
}

// ------------------------------------------------------------------------------ re-rank
// a value of a token held by pool/tail `sz` at index `si` (buffer buf), channel c
__device__ __forceinline__ const uint8_t* tk_src_tile(const TokState& s, int layer, int buf, int u, int sz, int si) {
  if (sz == TK_TAIL) return s.tail + (tk_tail_tok_index(s, layer, buf, u) / 16 + si / 16) * (long long)s.g.bf_tile();
  return s.pool[sz] + (tk_pool_tile_index(s, sz, layer, buf, u) + si / 16) * (long long)tk_tile_bytes(s, sz);
}

__device__ __forceinline__ unsigned tk_code_at(const TokGeo& g, const uint8_t* tile, int b, int row, int c, bool value) {
  const CodePos cp = value ? tk_vcode_pos(g, b, row, c) : tk_kcode_pos(g, b, row, c);
  const unsigned w = *reinterpret_cast<const unsigned*>(tile + cp.byte);
  return (w >> cp.bit) & ((1u << b) - 1u);
}

__device__ __forceinline__ float tk_value_at(const TokState& s, const uint8_t* tile, int sz, int row, int c, bool value) {
  const Geo g16{s.g.D, 16};
  if (sz == TK_BF16 || sz == TK_TAIL) {
    const int off = value ? bf16_v_off(g16, row, c) : bf16_k_off(g16, row, c);
    return __uint_as_float((unsigned)*reinterpret_cast<const uint16_t*>(tile + off) << 16);
  }
  const int b = tk_bits(sz);
  const unsigned code = tk_code_at(s.g, tile, b, row, c, value);
  const float2 par = reinterpret_cast<const float2*>(tile + (value ? s.g.off_vpar(b) : s.g.off_kpar(b)))[row];
  if (sz == TK_NQ1) return fmaf(code ? TK_NQ1_C : -TK_NQ1_C, par.y, par.x);
  return fmaf((float)code, par.y, par.x);
}

// eq. (2) decision, as IEEE float32 division decides it (fast estimate, exact division within
// 1e-5 of a half-integer or for scales outside [1e-30, 1e30])
__device__ __forceinline__ unsigned tk_quant_code(float x, float z, float s, float levels) {
  if (s == 0.f) return 0u;
  const float d = __fsub_rn(x, z);
  float qv = __fdividef(d, s);
  const float fr = qv - floorf(qv);
  if (fabsf(fr - 0.5f) < 1e-5f || !(s >= 1e-30f && s <= 1e30f)) qv = __fdiv_rn(d, s);
  qv = rintf(qv);
  qv = fminf(fmaxf(qv, 0.f), levels);
  return (unsigned)qv;
}

constexpr int TK_VROW = 129;   // padded row of the value buffer (floats), D <= 128

struct TkWarpBuf {
  uint8_t src[8192];     // the source tile last read (a BF16 tile of d = 128 is the largest)
  float vals[16 * TK_VROW];
  uint8_t codes[16 * 128];
  float2 par[16];
  int need[16];
  int src_id;            // (pool or tail) << 28 | tile index of src, -1 for none
  int pad[3];
};

template <int D>
__global__ void __launch_bounds__(TK_RERANK_THREADS, 1) tk_rerank_kernel(const TokState s, int layer0) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ unsigned hist[4][256];
  __shared__ unsigned long long pref[4];
  __shared__ long long need_rank[4];
  __shared__ int cut_mode[4];   // 0 select, 1 every key is past the cut, 2 no key is
  __shared__ int scan[4][TK_RERANK_THREADS];
  __shared__ int s_cnt[4];
  const int u = blockIdx.x, tid = threadIdx.x;
  const int layer = layer0 + (int)blockIdx.y;
  const long long su = (long long)blockIdx.y * s.units + u;   // scratch slot of (layer, unit)
  const TokLayer hd = s.hdr[layer];
  const int L = hd.L, nt = hd.n_tail, buf = hd.buf;
  const int4 c4 = *reinterpret_cast<const int4*>(s.cnt + ((long long)layer * s.units + u) * 4);
  const int cnt[4] = {c4.x, c4.y, c4.z, c4.w};
  int n_aged = nt - s.n_sink - s.n_recent;
  if (n_aged < 0) n_aged = 0;
  const int ncand = cnt[0] + cnt[1] + cnt[2] + cnt[3] + n_aged;
  const size_t mc = (size_t)s.max_context;
  unsigned long long* key = s.ckey + su * mc;
  int* src = s.csrc + su * mc;
  uint8_t* newt = s.newt + su * mc;
  int* src_of = s.src_of + su * mc;
  int* order = s.order + su * 4 * mc;
  // cut ranks (cumulative), double arithmetic without contraction as the host and oracle do
  long long cuts[4];
  {
    long long acc = 0;
    for (int z = 0; z < 4; ++z) {
      long long n = (long long)floor(__dmul_rn(s.frac[z], (double)L));
      if (z == 0) n -= s.n_sink + s.n_recent;
      if (n < 0) n = 0;
      acc += n;
      cuts[z] = acc;
    }
  }
  // ---- candidates
  for (int i = tid; i < L; i += TK_RERANK_THREADS) newt[i] = 0xFF;
  for (int i = tid; i < ncand; i += TK_RERANK_THREADS) {
    int z = 0, idx = i;
    while (z < 4 && idx >= cnt[z]) { idx -= cnt[z]; ++z; }
    int pos;
    float sc;
    if (z < 4) {
      const long long b = tk_pool_tok_index(s, z, layer, buf, u);
      pos = s.pos[z][b + idx];
      sc = s.score[z][b + idx];
    } else {
      z = TK_TAIL;
      idx += s.n_sink;
      const long long b = tk_tail_tok_index(s, layer, buf, u);
      pos = s.tail_pos[b + idx];
      sc = s.tail_score[b + idx];
    }
    key[i] = ((unsigned long long)(~__float_as_uint(fmaxf(sc, 0.f))) << 32) | (unsigned)pos;
    src[i] = (z << 28) | idx;
  }
  if (tid < 4) {
    const long long c = cuts[tid];
    cut_mode[tid] = c <= 0 ? 1 : (c >= ncand ? 2 : 0);
    pref[tid] = 0ull;
    need_rank[tid] = c - 1;
  }
  __syncthreads();
  // ---- the key at rank cuts[k] - 1, one radix digit (8 bits) per pass, all cuts at once
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 4 * 256; i += TK_RERANK_THREADS) hist[i >> 8][i & 255] = 0;
    __syncthreads();
    for (int i = tid; i < ncand; i += TK_RERANK_THREADS) {
      const unsigned long long kk = key[i];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (cut_mode[c] != 0) continue;
        const bool match = shift == 56 ? true : ((kk ^ pref[c]) >> (shift + 8)) == 0ull;
        if (match) atomicAdd(&hist[c][(kk >> shift) & 255u], 1u);
      }
    }
    __syncthreads();
    if (tid < 4 && cut_mode[tid] == 0) {
      long long r = need_rank[tid];
      int d = 0;
      for (; d < 256; ++d) {
        const long long h = hist[tid][d];
        if (r < h) break;
        r -= h;
      }
      if (d > 255) d = 255;
      pref[tid] |= (unsigned long long)d << shift;
      need_rank[tid] = r;
    }
    __syncthreads();
  }
  // ---- new tiers: the rank's tier, never above the current one
  for (int i = tid; i < ncand; i += TK_RERANK_THREADS) {
    const unsigned long long kk = key[i];
    int d = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) d += cut_mode[c] == 1 || (cut_mode[c] == 0 && kk > pref[c]);
    const int sr = src[i];
    const int z = sr >> 28;
    const int old = z == TK_TAIL ? TK_BF16 : z;
    const int nw = d > old ? d : old;
    const int pos = (int)(unsigned)kk;
    if (pos >= 0 && pos < L) {
      newt[pos] = (uint8_t)nw;
      src_of[pos] = sr;
    } else {
      atomicOr(s.err, ERR_TABLE);
    }
  }
  __syncthreads();
  // ---- positional order of every kept tier
  {
    const int chunk = (L + TK_RERANK_THREADS - 1) / TK_RERANK_THREADS;
    const int p0 = tid * chunk, p1 = p0 + chunk < L ? p0 + chunk : L;
    int c[4] = {0, 0, 0, 0};
    for (int q = p0; q < p1; ++q) {
      const int z = newt[q];
      if (z < 4) ++c[z];
    }
    for (int z = 0; z < 4; ++z) scan[z][tid] = c[z];
    __syncthreads();
    if (tid < 4) {
      int acc = 0;
      for (int i = 0; i < TK_RERANK_THREADS; ++i) {
        const int v = scan[tid][i];
        scan[tid][i] = acc;
        acc += v;
      }
      s_cnt[tid] = acc;
      if (acc > s.cap[tid]) atomicOr(s.err, ERR_CAPACITY);
    }
    __syncthreads();
    int o[4] = {scan[0][tid], scan[1][tid], scan[2][tid], scan[3][tid]};
    for (int q = p0; q < p1; ++q) {
      const int z = newt[q];
      if (z < 4) {
        if (o[z] < s.cap[z]) order[z * mc + o[z]] = q;
        ++o[z];
      }
    }
  }
  __syncthreads();
  if (tid < 4) s.ncnt[su * 4 + tid] = s_cnt[tid] < s.cap[tid] ? s_cnt[tid] : s.cap[tid];
}

// stage source tile `id` ((pool or tail) << 28 | tile) of unit u in the warp's shared buffer
__device__ __forceinline__ const uint8_t* tk_stage(TkWarpBuf& W, const TokState& s, int layer, int buf, int u, int id,
                                                   int lane) {
  if (W.src_id != id) {
    __syncwarp();
    const int sz = id >> 28, ti = id & 0x0FFFFFFF;
    const uint8_t* g = tk_src_tile(s, layer, buf, u, sz, ti * 16);
    const int bytes = tk_tile_bytes(s, sz);
    // every lane's pieces in flight at once: one memory latency per staged tile
    for (int off = lane * 16; off < bytes; off += 512) cp_async16(W.src + off, g + off);
    cp_async_commit();
    cp_async_wait_all();
    __syncwarp();
    if (lane == 0) W.src_id = id;
    __syncwarp();
  }
  return W.src;
}

// byte offset (in the tile) and bit of the code of token `tok`, channel c, in a B-bit tile
template <int D, int B>
__device__ __forceinline__ void tk_code_loc(int tok, int c, bool value, int& byte, int& bit) {
  constexpr int PW = 4 / B, WPL = D * B / 64, CW = WPL < 4 ? WPL : 4;
  const int step = c >> 4;
  const int row16 = value ? (c & 15) : tok, col16 = value ? tok : (c & 15);
  const int ln = (row16 & 7) * 4 + ((col16 & 7) >> 1);
  const int reg = (row16 >> 3) + 2 * (col16 >> 3);
  const int j = step / PW, k = step % PW;
  byte = ((j / CW) * 32 + ln) * (CW * 4) + (j % CW) * 4 + (value ? 2 * D * B : 0);
  bit = 16 * (col16 & 1) + B * (4 * k + reg);
}

template <int D, int B>
__device__ __forceinline__ unsigned tk_code_t(const uint8_t* tile, int tok, int c, bool value) {
  int byte, bit;
  tk_code_loc<D, B>(tok, c, value, byte, bit);
  return (*reinterpret_cast<const unsigned*>(tile + byte) >> bit) & ((1u << B) - 1u);
}

// the value a B-bit tile (normal for the 1-bit tier) reconstructs: one float32 fma
template <int D, int B>
__device__ __forceinline__ float tk_value_t(const uint8_t* tile, int tok, int c, bool value) {
  const unsigned code = tk_code_t<D, B>(tile, tok, c, value);
  const float2 par = reinterpret_cast<const float2*>(tile + 4 * D * B + (value ? 128 : 0))[tok];
  if (B == 1) return fmaf(code ? TK_NQ1_C : -TK_NQ1_C, par.y, par.x);
  return fmaf((float)code, par.y, par.x);
}

// Field masks of the code words (layout in qe_tok.cuh): key side, the fields of row rr (0: row
// g, 1: row g + 8) of lane 4 g + t; value side, the fields of token 2 t + hf + 8 rb.
template <int B>
__host__ __device__ constexpr unsigned tk_kmask(int rr) {
  unsigned m = 0u;
  for (int hf = 0; hf < 2; ++hf)
    for (int k = 0; k < 4 / B; ++k)
      for (int q = 0; q < 2; ++q) m |= ((1u << B) - 1u) << (16 * hf + B * (4 * k + rr + 2 * q));
  return m;
}
template <int B>
__host__ __device__ constexpr unsigned tk_vmask(int hf, int rb) {
  unsigned m = 0u;
  for (int k = 0; k < 4 / B; ++k)
    for (int q = 0; q < 2; ++q) m |= ((1u << B) - 1u) << (16 * hf + B * (4 * k + 2 * rb + q));
  return m;
}

// Mean and population std of one row of D float32 values in shared memory (HqeKV reading notes,
// §2.3 eq. (3)), each the exact value rounded once to float32 (qe_exact_stats.cuh).  Every lane
// turns its D / 32 values into integers at the row's scale and the warp adds the integer sums;
// a row whose nonzero values span more than the fast path's window goes to the wide path on
// lane 0.  Every lane returns the same m and sd.
template <int D>
__device__ __forceinline__ void tk_row_mean_std(const float* x, int lane, float& m, float& sd) {
  constexpr int NV = D / 32, LGD = D == 128 ? 7 : 6;
  float v[NV];
  unsigned E = 0u;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    v[i] = x[lane + 32 * i];
    const xs::Parts pt = xs::parts(v[i]);
    if (pt.mant && (unsigned)pt.ee > E) E = (unsigned)pt.ee;
  }
  E = __reduce_max_sync(0xffffffffu, E);
  if (E == 0u) {   // all zeros
    m = 0.f;
    sd = 0.f;
    return;
  }
  xs::FastAcc a{0, 0, 0};
#pragma unroll
  for (int i = 0; i < NV; ++i) xs::fast_add(a, v[i], (int)E);
  if (__any_sync(0xffffffffu, a.bad)) {
    float mw = 0.f, sw = 0.f;
    if (lane == 0) {
      xs::WideAcc w;
      xs::wide_zero(w);
      for (int c = 0; c < D; ++c) xs::wide_acc(w, x[c]);
      xs::wide_finish(w, LGD, mw, sw);
    }
    m = __shfl_sync(0xffffffffu, mw, 0);
    sd = __shfl_sync(0xffffffffu, sw, 0);
    return;
  }
  long long S = a.s;
  unsigned long long qlo = (unsigned long long)a.q, qhi = (unsigned long long)(a.q >> 64);
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    S += __shfl_xor_sync(0xffffffffu, S, o);
    const unsigned long long lo2 = __shfl_xor_sync(0xffffffffu, qlo, o);
    const unsigned long long hi2 = __shfl_xor_sync(0xffffffffu, qhi, o);
    const xs::u128 sum = (((xs::u128)qhi << 64) | qlo) + (((xs::u128)hi2 << 64) | lo2);
    qlo = (unsigned long long)sum;
    qhi = (unsigned long long)(sum >> 64);
  }
  xs::fast_finish(S, ((xs::u128)qhi << 64) | qlo, (int)E, LGD, m, sd);
}

// Rows of one destination tile of the B-bit tier (1-bit: the normal quantizer).  Rows that keep
// their tier move word-wise: a row's fields sit in fixed lanes and bit positions, so moving it
// from source row s to destination row d is a mask, a shift and an or per code word.  Rows
// arriving from another tier are re-quantized from the values it held.  Lane r < 16 holds row
// r's source (my_sz, my_si, my_id); `valid` marks rows present.
template <int D, int B>
__device__ void tk_rebuild_qtile(const TokState& s, int layer, int buf, int u, TkWarpBuf& W, uint8_t* dst,
                                 unsigned valid, int my_sz, int my_si, int my_id, int lane) {
  constexpr int Z = B == 4 ? TK_INT4 : B == 2 ? TK_INT2 : TK_NQ1;
  constexpr float LEVELS = (float)((1 << B) - 1);
  constexpr int WPL = D * B / 64, CW = WPL < 4 ? WPL : 4, PW = 4 / B;
  const Geo g16{D, 16};
  const int g = lane >> 2, t = lane & 3;
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {   // keys, then values
    const bool value = half == 1;
    const int NT = value ? 4 : 2;           // tokens whose fields this lane's words hold
    int tok[4], tid[4], tsi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      tok[i] = value ? 2 * t + (i & 1) + 8 * (i >> 1) : g + 8 * (i & 1);
      tid[i] = __shfl_sync(0xffffffffu, my_id, tok[i]);
      tsi[i] = __shfl_sync(0xffffffffu, my_si, tok[i]);
    }
    if (lane < 16) W.need[lane] = my_id >= 0 && my_sz != Z;
    if (lane < 16 && my_id < 0) W.par[lane] = make_float2(0.f, 0.f);
    unsigned word[WPL];
#pragma unroll
    for (int j = 0; j < WPL; ++j) word[j] = 0u;
    const int boff = value ? 2 * D * B : 0;
    // 1. gather, one staged source tile at a time
    unsigned todo = valid;
    while (todo) {
      const int id = __shfl_sync(0xffffffffu, my_id, __ffs(todo) - 1);
      const unsigned grp = __ballot_sync(0xffffffffu, my_id == id) & todo;
      const uint8_t* st = tk_stage(W, s, layer, buf, u, id, lane);
      const int sz = id >> 28;
      if (sz == Z) {
        // word-wise moves of this lane's rows that come from the staged tile
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i >= NT || tid[i] != id) continue;
          const int sr = tsi[i] & 15;
          int src_lane, sh;
          unsigned mask;
          if (!value) {
            src_lane = 4 * (sr & 7) + t;
            mask = (sr >> 3) ? tk_kmask<B>(1) : tk_kmask<B>(0);
            sh = B * (i - (sr >> 3));
          } else {
            src_lane = 4 * g + ((sr & 7) >> 1);
            const int hf_s = sr & 1, rb_s = sr >> 3;
            mask = hf_s ? (rb_s ? tk_vmask<B>(1, 1) : tk_vmask<B>(1, 0)) : (rb_s ? tk_vmask<B>(0, 1) : tk_vmask<B>(0, 0));
            sh = 16 * ((i & 1) - hf_s) + 2 * B * ((i >> 1) - rb_s);
          }
#pragma unroll
          for (int j = 0; j < WPL; ++j) {
            const unsigned sw = *reinterpret_cast<const unsigned*>(st + boff + ((j / CW) * 32 + src_lane) * (CW * 4) +
                                                                   (j % CW) * 4) & mask;
            word[j] |= sh >= 0 ? sw << sh : sw >> (-sh);
          }
        }
        if (lane < 16 && my_id == id)
          W.par[lane] = reinterpret_cast<const float2*>(st + 4 * D * B + (value ? 128 : 0))[my_si & 15];
      } else {
        for (unsigned m = grp; m; m &= m - 1) {
          const int row = __ffs(m) - 1;
          const int srow = __shfl_sync(0xffffffffu, my_si, row) & 15;
          if (sz == TK_BF16 || sz == TK_TAIL) {
#pragma unroll
            for (int c = lane; c < D; c += 32) {
              const int off = value ? bf16_v_off(g16, srow, c) : bf16_k_off(g16, srow, c);
              W.vals[row * TK_VROW + c] = __uint_as_float((unsigned)*reinterpret_cast<const uint16_t*>(st + off) << 16);
            }
          } else if (sz == TK_INT4) {
#pragma unroll
            for (int c = lane; c < D; c += 32) W.vals[row * TK_VROW + c] = tk_value_t<D, 4>(st, srow, c, value);
          } else {   // 2-bit (a token only moves down, so a 1-bit source never reaches another tier)
#pragma unroll
            for (int c = lane; c < D; c += 32) W.vals[row * TK_VROW + c] = tk_value_t<D, 2>(st, srow, c, value);
          }
        }
      }
      todo &= ~grp;
    }
    __syncwarp();
    // 2. quantize the rows arriving from another tier
    if (B == 1) {
      // eqs. (3)-(4), b = 1: the row's exact mean and population std, each rounded once to
      // float32; code 1 where x > mean (all zeros when the std is 0)
      for (int row = 0; row < 16; ++row) {
        if (!W.need[row]) continue;
        const float* x = W.vals + row * TK_VROW;
        float m, sd;
        tk_row_mean_std<D>(x, lane, m, sd);
#pragma unroll
        for (int c = lane; c < D; c += 32) W.codes[row * 128 + c] = (uint8_t)(sd > 0.f && x[c] > m);
        if (lane == 0) W.par[row] = make_float2(m, sd);
      }
    } else {
      // eq. (2) per token: z = min, s = (max - min) / (2^b - 1) in float32
      for (int row = 0; row < 16; ++row) {
        if (!W.need[row]) continue;
        float mn = INFINITY, mx = -INFINITY;
#pragma unroll
        for (int c = lane; c < D; c += 32) {
          const float x = W.vals[row * TK_VROW + c];
          mn = fminf(mn, x);
          mx = fmaxf(mx, x);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        const float sc = __fdiv_rn(__fsub_rn(mx, mn), LEVELS);
#pragma unroll
        for (int c = lane; c < D; c += 32)
          W.codes[row * 128 + c] = (uint8_t)tk_quant_code(W.vals[row * TK_VROW + c], mn, sc, LEVELS);
        if (lane == 0) W.par[row] = make_float2(mn, sc);
      }
    }
    __syncwarp();
    // 3. the fields of this lane's re-quantized tokens, then the words and the parameters
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i >= NT || !W.need[tok[i]]) continue;
      const int tk = tok[i];
#pragma unroll
      for (int j = 0; j < WPL; ++j)
#pragma unroll
        for (int kk = 0; kk < PW; ++kk) {
          const int step = j * PW + kk;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            if (!value) {   // row tk = g + 8 i: registers r = i + 2 q, both halves
              const int r = i + 2 * q;
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                const int ch = 16 * step + 2 * t + hf + 8 * q;
                word[j] |= (unsigned)W.codes[tk * 128 + ch] << (16 * hf + B * (4 * kk + r));
              }
            } else {        // token tk = 2 t + hf + 8 rb: registers r = 2 rb + q (rows g + 8 q), half hf
              const int hf = i & 1, r = 2 * (i >> 1) + q;
              const int ch = 16 * step + g + 8 * q;
              word[j] |= (unsigned)W.codes[tk * 128 + ch] << (16 * hf + B * (4 * kk + r));
            }
          }
        }
    }
    uint8_t* blk = dst + boff;
#pragma unroll
    for (int j = 0; j < WPL; ++j)
      *reinterpret_cast<unsigned*>(blk + ((j / CW) * 32 + lane) * (CW * 4) + (j % CW) * 4) = word[j];
    if (lane < 16) reinterpret_cast<float2*>(dst + 4 * D * B + (value ? 128 : 0))[lane] = W.par[lane];
    __syncwarp();
  }
}

// Rebuild of one unit's pools and tail in the other buffer after tk_rerank_kernel chose the new
// tiers: TK_REBUILD_SPLIT CTAs per unit share its destination tiles, one tile per warp at a time.
// A destination tile's rows (position order) come from few source tiles: the warp stages each
// distinct source tile once in shared memory and serves every row that reads from it.
constexpr int TK_REBUILD_SPLIT = 9;
// six warps per CTA: two CTAs fit on an SM (shared memory: six warp buffers each)
constexpr int TK_REBUILD_WARPS = 6;
constexpr int TK_REBUILD_THREADS = TK_REBUILD_WARPS * 32;

template <int D>
__global__ void __launch_bounds__(TK_REBUILD_THREADS, 2) tk_rebuild_kernel(const TokState s, int layer0) {
  extern __shared__ __align__(1024) uint8_t smem[];
  TkWarpBuf* wb = reinterpret_cast<TkWarpBuf*>(smem);
  const int u = blockIdx.x / TK_REBUILD_SPLIT, part = blockIdx.x - u * TK_REBUILD_SPLIT;
  const int layer = layer0 + (int)blockIdx.y;
  const long long su = (long long)blockIdx.y * s.units + u;   // scratch slot of (layer, unit)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wall = part * TK_REBUILD_WARPS + warp, nwall = TK_REBUILD_SPLIT * TK_REBUILD_WARPS;
  const TokGeo geo = s.g;
  const Geo g16{D, 16};
  const TokLayer hd = s.hdr[layer];
  const int nt = hd.n_tail, buf = hd.buf, nb = buf ^ 1;
  int n_aged = nt - s.n_sink - s.n_recent;
  if (n_aged < 0) n_aged = 0;
  const size_t mc = (size_t)s.max_context;
  const int* order = s.order + su * 4 * mc;
  const int* src_of = s.src_of + su * mc;
  const bool reset = s.score_window > 0;
  int ncnt[4];
  for (int z = 0; z < 4; ++z) ncnt[z] = s.ncnt[su * 4 + z];
  TkWarpBuf& W = wb[warp];
  if (lane == 0) W.src_id = -1;
  __syncwarp();
  const int T0 = (ncnt[0] + 15) >> 4, T1 = (ncnt[1] + 15) >> 4, T2 = (ncnt[2] + 15) >> 4, T3 = (ncnt[3] + 15) >> 4;
  const int Ttot = T0 + T1 + T2 + T3;
  for (int tt = wall; tt < Ttot; tt += nwall) {
    int z, kt;
    if (tt < T0) { z = 0; kt = tt; }
    else if (tt < T0 + T1) { z = 1; kt = tt - T0; }
    else if (tt < T0 + T1 + T2) { z = 2; kt = tt - T0 - T1; }
    else { z = 3; kt = tt - T0 - T1 - T2; }
    const long long pb = tk_pool_tok_index(s, z, layer, nb, u);
    uint8_t* dst = s.pool[z] + (tk_pool_tile_index(s, z, layer, nb, u) + kt) * (long long)tk_tile_bytes(s, z);
    // lane r < 16: row r's source (pool or tail, index) and its tile id; positions and scores
    int my_sz = -1, my_si = 0, my_id = -1;
    if (lane < 16) {
      const int idx = 16 * kt + lane;
      if (idx < ncnt[z]) {
        const int q = order[z * mc + idx];
        const int sr = src_of[q];
        my_sz = sr >> 28;
        my_si = sr & 0x0FFFFFFF;
        my_id = (my_sz << 28) | (my_si >> 4);
        float sc = 0.f;
        if (!reset) {
          sc = my_sz == TK_TAIL ? s.tail_score[tk_tail_tok_index(s, layer, buf, u) + my_si]
                                : s.score[my_sz][tk_pool_tok_index(s, my_sz, layer, buf, u) + my_si];
        }
        s.pos[z][pb + idx] = q;
        s.score[z][pb + idx] = sc;
      }
    }
    const unsigned valid = __ballot_sync(0xffffffffu, my_id >= 0);
    if (z == 0) {
      // BF16 -> BF16: rows move to their new places (empty rows become zeros)
      unsigned todo = valid;
      while (todo) {
        const int id = __shfl_sync(0xffffffffu, my_id, __ffs(todo) - 1);
        const unsigned grp = __ballot_sync(0xffffffffu, my_id == id) & todo;
        const uint8_t* st = tk_stage(W, s, layer, buf, u, id, lane);
        for (unsigned m = grp; m; m &= m - 1) {
          const int row = __ffs(m) - 1;
          const int srow = __shfl_sync(0xffffffffu, my_si, row) & 15;
          for (int c = 2 * lane; c < D; c += 64) {
            *reinterpret_cast<unsigned*>(dst + bf16_k_off(g16, row, c)) =
                *reinterpret_cast<const unsigned*>(st + bf16_k_off(g16, srow, c));
            *reinterpret_cast<uint16_t*>(dst + bf16_v_off(g16, row, c)) =
                *reinterpret_cast<const uint16_t*>(st + bf16_v_off(g16, srow, c));
            *reinterpret_cast<uint16_t*>(dst + bf16_v_off(g16, row, c + 1)) =
                *reinterpret_cast<const uint16_t*>(st + bf16_v_off(g16, srow, c + 1));
          }
        }
        todo &= ~grp;
      }
      for (unsigned m = ~valid & 0xFFFFu; m; m &= m - 1) {
        const int row = __ffs(m) - 1;
        for (int c = 2 * lane; c < D; c += 64) {
          *reinterpret_cast<unsigned*>(dst + bf16_k_off(g16, row, c)) = 0u;
          *reinterpret_cast<uint16_t*>(dst + bf16_v_off(g16, row, c)) = 0;
          *reinterpret_cast<uint16_t*>(dst + bf16_v_off(g16, row, c + 1)) = 0;
        }
      }
      __syncwarp();
      continue;
    }
    if (z == TK_INT4) tk_rebuild_qtile<D, 4>(s, layer, buf, u, W, dst, valid, my_sz, my_si, my_id, lane);
    else if (z == TK_INT2) tk_rebuild_qtile<D, 2>(s, layer, buf, u, W, dst, valid, my_sz, my_si, my_id, lane);
    else tk_rebuild_qtile<D, 1>(s, layer, buf, u, W, dst, valid, my_sz, my_si, my_id, lane);
  }
  // ---- the new tail: the sink and the recent tokens, moved up over the aged ones
  {
    const int ntn = nt - n_aged;
    const long long ob = tk_tail_tok_index(s, layer, buf, u), nbb = tk_tail_tok_index(s, layer, nb, u);
    const int tiles = (ntn + 15) >> 4;
    for (int tt = wall; tt < tiles; tt += nwall) {
      uint8_t* dst = s.tail + (nbb / 16 + tt) * (long long)geo.bf_tile();
      for (int row = 0; row < 16; ++row) {
        const int i = 16 * tt + row;
        const bool valid = i < ntn;
        const int si = i < s.n_sink ? i : i + n_aged;
        const uint8_t* st = s.tail + (ob / 16 + si / 16) * (long long)geo.bf_tile();
        const int srow = si & 15;
        for (int c = 2 * lane; c < D; c += 64) {
          unsigned kk = 0u;
          uint16_t v0 = 0, v1 = 0;
          if (valid) {
            kk = *reinterpret_cast<const unsigned*>(st + bf16_k_off(g16, srow, c));
            v0 = *reinterpret_cast<const uint16_t*>(st + bf16_v_off(g16, srow, c));
            v1 = *reinterpret_cast<const uint16_t*>(st + bf16_v_off(g16, srow, c + 1));
          }
          *reinterpret_cast<unsigned*>(dst + bf16_k_off(g16, row, c)) = kk;
          *reinterpret_cast<uint16_t*>(dst + bf16_v_off(g16, row, c)) = v0;
          *reinterpret_cast<uint16_t*>(dst + bf16_v_off(g16, row, c + 1)) = v1;
        }
        if (lane == 0 && valid) {
          s.tail_pos[nbb + i] = s.tail_pos[ob + si];
          s.tail_score[nbb + i] = reset ? 0.f : s.tail_score[ob + si];
        }
      }
    }
  }
}

// After the re-rank of a layer: cost prefix of the new counts and the header switch.
__global__ void tk_finish_kernel(TokState s, int layer0) {
  __shared__ long long part[256];
  const int tid = threadIdx.x;
  const int layer = layer0 + (int)blockIdx.y;
  int* cnt = s.cnt + (long long)layer * s.units * 4;
  const int* ncnt = s.ncnt + (long long)blockIdx.y * s.units * 4;
  for (int i = tid; i < s.units * 4; i += 256) cnt[i] = ncnt[i];
  __syncthreads();
  long long* cum = s.cum + (long long)layer * (s.units + 1);
  // each thread sums a contiguous run of units, then a serial prefix over the threads
  const int per = (s.units + 255) / 256;
  const int u0 = tid * per, u1 = u0 + per < s.units ? u0 + per : s.units;
  long long acc = 0;
  for (int u = u0; u < u1; ++u)
    for (int z = 0; z < 4; ++z) acc += (long long)s.cost[z] * ((cnt[u * 4 + z] + 15) >> 4);
  part[tid] = acc;
  __syncthreads();
  if (tid == 0) {
    long long run = 0;
    for (int i = 0; i < 256; ++i) {
      const long long v = part[i];
      part[i] = run;
      run += v;
    }
  }
  __syncthreads();
  long long run = part[tid];
  for (int u = u0; u < u1; ++u) {
    cum[u] = run;
    for (int z = 0; z < 4; ++z) run += (long long)s.cost[z] * ((cnt[u * 4 + z] + 15) >> 4);
  }
  if (u1 == s.units && u0 < u1) cum[s.units] = run;
  if (s.units == 0 && tid == 0) cum[0] = 0;
  __syncthreads();
  if (tid == 0) {
    TokLayer& hd = s.hdr[layer];
    int n_aged = hd.n_tail - s.n_sink - s.n_recent;
    if (n_aged < 0) n_aged = 0;
    hd.n_tail -= n_aged;
    hd.buf ^= 1;
    hd.step = 0;
  }
}

// ------------------------------------------------------------------------------ launchers
size_t tk_rerank_smem(int /*D*/) { return (size_t)TK_REBUILD_WARPS * sizeof(TkWarpBuf); }

template <int D>
static cudaError_t tk_prepare_t() {
  constexpr int STAGE = 64 * D;
  constexpr int NST = TK_STAGE_TOTAL / (TK_WARPS * STAGE) < 4 ? TK_STAGE_TOTAL / (TK_WARPS * STAGE) : 4;
  cudaError_t e = cudaFuncSetAttribute(tk_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TK_WARPS * NST * STAGE);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tk_rebuild_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tk_rerank_smem(D));
}

cudaError_t tk_prepare(int D) { return D == 128 ? tk_prepare_t<128>() : tk_prepare_t<64>(); }

int tk_attn_warps() { return TK_WARPS; }

cudaError_t tk_launch_append1(const TokState& s, int layer, const uint16_t* k, const uint16_t* v, cudaStream_t st) {
  tk_append1_kernel<<<s.units, s.g.D / 2, 0, st>>>(s, layer, k, v);
  return cudaGetLastError();
}

cudaError_t tk_launch_append(const TokState& s, int layer, int n, bool prefill, const uint16_t* k, const uint16_t* v,
                             int n_sm, cudaStream_t st) {
  const long long total = (long long)s.units * n * (s.g.D / 2);
  long long blocks = (total + 255) / 256;
  if (blocks > (long long)n_sm * 16) blocks = (long long)n_sm * 16;
  if (blocks < 1) blocks = 1;
  tk_append_kernel<<<(int)blocks, 256, 0, st>>>(s, layer, n, prefill ? 1 : 0, k, v);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  tk_commit_kernel<<<1, 32, 0, st>>>(s, layer, n, prefill ? 1 : 0);
  return cudaGetLastError();
}

__global__ void tk_commit_pending_kernel(TokState s, int layer, int pend) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    s.hdr[layer].L += pend;
    s.hdr[layer].n_tail += pend;
  }
}

cudaError_t tk_launch_commit_pending(const TokState& s, int layer, int pend, cudaStream_t st) {
  tk_commit_pending_kernel<<<1, 32, 0, st>>>(s, layer, pend);
  return cudaGetLastError();
}

cudaError_t tk_launch_attn(const TokState& s, int layer, int pend, const uint16_t* knew, const uint16_t* vnew,
                           const uint16_t* q, float scale_log2, float* part_o, float2* part_ml, float* logits, int lg_cap,
                           int grid, cudaStream_t st, int debug_expire) {
  const int D = s.g.D;
  TkAttnArgs a;
  a.st = s;
  a.layer = layer;
  a.pend = pend;
  a.knew = pend > 0 ? knew : nullptr;
  a.vnew = pend > 0 ? vnew : nullptr;
  a.q = q;
  a.scale_log2 = scale_log2;
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.logits = logits;
  a.lg_cap = lg_cap;
  a.debug_expire = debug_expire;
  const int stage = 64 * D;
  const int nst = TK_STAGE_TOTAL / (TK_WARPS * stage) < 4 ? TK_STAGE_TOTAL / (TK_WARPS * stage) : 4;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TK_WARPS * 32);
  cfg.dynamicSmemBytes = (size_t)TK_WARPS * nst * stage;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128) return cudaLaunchKernelEx(&cfg, tk_attn_kernel<128>, a);
  return cudaLaunchKernelEx(&cfg, tk_attn_kernel<64>, a);
}

// programmatic dependent of the attention launch before it on the stream
cudaError_t tk_launch_merge(const TokState& s, int layer, int pend, const float* part_o, const float2* part_ml,
                            const float* logits, int lg_cap, int grid, void* out, int out_fp32, cudaStream_t st) {
  TkMergeArgs m;
  m.st = s;
  m.layer = layer;
  m.pend = pend;
  m.NW = grid * TK_WARPS;
  m.part_o = part_o;
  m.part_ml = part_ml;
  m.logits = logits;
  m.lg_cap = lg_cap;
  m.out = out;
  m.out_fp32 = out_fp32;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(s.units * TK_MERGE_SPLIT);
  cfg.blockDim = dim3(TK_MERGE_THREADS);
  cfg.dynamicSmemBytes = (size_t)s.G * (m.NW + 2) * sizeof(float);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (s.g.D == 128) return cudaLaunchKernelEx(&cfg, tk_merge_kernel<128>, m);
  return cudaLaunchKernelEx(&cfg, tk_merge_kernel<64>, m);
}

cudaError_t tk_launch_rerank(const TokState& s, int layer0, int n_layers, cudaStream_t st) {
  const size_t sm = tk_rerank_smem(s.g.D);
  const dim3 sel(s.units, n_layers), reb(s.units * TK_REBUILD_SPLIT, n_layers), fin(1, n_layers);
  if (s.g.D == 128) tk_rerank_kernel<128><<<sel, TK_RERANK_THREADS, 0, st>>>(s, layer0);
  else tk_rerank_kernel<64><<<sel, TK_RERANK_THREADS, 0, st>>>(s, layer0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (s.g.D == 128) tk_rebuild_kernel<128><<<reb, TK_REBUILD_THREADS, sm, st>>>(s, layer0);
  else tk_rebuild_kernel<64><<<reb, TK_REBUILD_THREADS, sm, st>>>(s, layer0);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  tk_finish_kernel<<<fin, 256, 0, st>>>(s, layer0);
  return cudaGetLastError();
}

}  // namespace qe
