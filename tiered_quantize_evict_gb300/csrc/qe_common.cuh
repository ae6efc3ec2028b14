// qe_common.cuh -- device state layout, fragment-native tile layouts and PTX wrappers.
//
// Window slots are stored in the exact register order the m16n8k16 tensor-core
// fragments want, so the attention kernel moves a whole tile into shared
// memory with one bulk copy and each lane then reads its operands with
// conflict-free 16-byte loads (no ldmatrix, no swizzle, no shuffles).
//
// bf16 window slot (4 w d bytes): w/16 sub-tiles of 16 tokens; each sub-tile
// holds the key fragments (d/16 of 512 B, A operand of Q K^T with tokens as
// rows) followed by the value fragments (d/16 of 512 B, A operand of V^T P^T
// with channels as rows).
//
// 2-bit window slot: key codes (w d / 4 B), key min[d], key scale[d], then value
// codes (w d / 4 B), value min[w], value scale[w] (float32; the parameter arrays
// are permuted so each lane reads its own as 16-byte vectors).  Codes
// are grouped per lane in 32-bit words; a word carries two fragments of 8
// codes: fragment f, register r (R = 4 f + r), element e sits at bit 2 R + 16 e.
// Shifting the word by 8 - 2R brings the register's two codes to bits 8 and 24,
// and one and-or with 0x03000300 / 0x3C003C00 makes them the f16 pair
// (1 + code / 4) the tensor core consumes; the constant 1 is removed through
// the key bias and the value offset.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#ifndef QE_HD
#define QE_HD __host__ __device__ __forceinline__
#endif

namespace qe {

enum : int { TIER_NONE = 0, TIER_PINNED = 1, TIER_FULL = 2, TIER_QUANT = 3, TIER_EVICTED = 4 };

// routing counters per layer: routes, first packs, ledger reuses, promotions, evictions, and
// promotions / re-demotions that took their previous slot back (no host transfer)
constexpr int N_STATS = 8;

enum : unsigned { ERR_FREELIST = 1u, ERR_TABLE = 2u, ERR_TIMEOUT = 4u, ERR_COUNT = 8u, ERR_MOVES = 16u,
                  ERR_CAPACITY = 32u };

// ---------------------------------------------------------------------------- geometry
struct Geo {
  int D, W;
  QE_HD int sub_tiles() const { return W / 16; }
  QE_HD int sub_bytes() const { return 64 * D; }                 // 16 tokens, K + V, bf16
  QE_HD int bslot_bytes() const { return 4 * W * D; }
  QE_HD int kcode_bytes() const { return W * D / 4; }
  QE_HD int qslot_bytes() const { return 2 * (W * D / 4) + 8 * D + 8 * W; }
  QE_HD int wpl() const { return (W / 16) * (D / 16) / 2; }       // code words per lane (K or V)
  QE_HD int cw() const { return wpl() < 4 ? wpl() : 4; }          // words per lane per chunk
  // 2-bit slot: the key half (codes, min[D], scale[D]) then the value half (codes, min[W],
  // scale[W]); each half is one contiguous 16-byte-aligned block
  QE_HD int khalf_bytes() const { return kcode_bytes() + 8 * D; }
  QE_HD int vhalf_bytes() const { return kcode_bytes() + 8 * W; }
  QE_HD int off_kmin() const { return kcode_bytes(); }
  QE_HD int off_kscale() const { return kcode_bytes() + 4 * D; }
  QE_HD int off_vcode() const { return khalf_bytes(); }
  QE_HD int off_vmin() const { return khalf_bytes() + kcode_bytes(); }
  QE_HD int off_vscale() const { return khalf_bytes() + kcode_bytes() + 4 * W; }
};

// byte offset of K[r][c] inside a bf16 slot (r < W)
QE_HD int bf16_k_off(const Geo& g, int r, int c) {
  int sub = r >> 4, rr = r & 15, ks = c >> 4, ci = c & 15;
  int lane = (rr & 7) * 4 + ((ci & 7) >> 1);
  int reg = (rr >> 3) + 2 * (ci >> 3);
  return sub * g.sub_bytes() + ks * 512 + lane * 16 + reg * 4 + (ci & 1) * 2;
}
// byte offset of V[r][c] inside a bf16 slot
QE_HD int bf16_v_off(const Geo& g, int r, int c) {
  int sub = r >> 4, rt = r & 15, mc = c >> 4, rc = c & 15;
  int lane = (rc & 7) * 4 + ((rt & 7) >> 1);
  int reg = (rc >> 3) + 2 * (rt >> 3);
  return sub * g.sub_bytes() + 32 * g.D + mc * 512 + lane * 16 + reg * 4 + (rt & 1) * 2;
}

// (byte offset of the 32-bit word, bit position) of a code inside the K or V code block
struct CodePos { int byte; int bit; };
QE_HD CodePos code_word(const Geo& g, int F, int lane, int reg, int e) {
  int wi = F >> 1, f = F & 1;
  int cw = g.cw();
  CodePos p;
  p.byte = ((wi / cw) * 32 + lane) * (cw * 4) + (wi % cw) * 4;
  p.bit = 8 * f + 2 * reg + 16 * e;
  return p;
}
// key code of token r, channel c (fragments ordered token-tile major, channel-step minor)
QE_HD CodePos kcode_pos(const Geo& g, int r, int c) {
  int mt = r >> 4, rr = r & 15, ks = c >> 4, ci = c & 15;
  int lane = (rr & 7) * 4 + ((ci & 7) >> 1);
  int reg = (rr >> 3) + 2 * (ci >> 3);
  return code_word(g, mt * (g.D / 16) + ks, lane, reg, ci & 1);
}
// value code of token r, channel c (A = V^T: fragments ordered channel-tile major, token-step minor)
QE_HD CodePos vcode_pos(const Geo& g, int r, int c) {
  int mc = c >> 4, rc = c & 15, kt = r >> 4, rt = r & 15;
  int lane = (rc & 7) * 4 + ((rt & 7) >> 1);
  int reg = (rc >> 3) + 2 * (rt >> 3);
  CodePos p = code_word(g, mc * (g.W / 16) + kt, lane, reg, rt & 1);
  p.byte += g.off_vcode();
  return p;
}

// Inverse of kcode_pos / vcode_pos: the (token r, channel c) whose code sits at bit
// 8 f + 2 reg + 16 e of word widx of the key code block (value = false) or of the value code
// block (value = true; widx counted from the start of that block).
struct RC { int r, c; };
QE_HD RC code_rc(const Geo& g, bool value, int widx, int reg, int f, int e) {
  const int cw = g.cw();
  const int chunk = widx / (32 * cw), rem = widx - chunk * 32 * cw;
  const int lane = rem / cw, wi = chunk * cw + (rem - lane * cw);
  const int F = 2 * wi + f;
  const int a = (lane >> 2) + 8 * (reg & 1);              // row inside the 16 x 16 fragment
  const int b = ((lane & 3) << 1) + e + 8 * (reg >> 1);   // column inside the fragment
  RC o;
  if (!value) {
    const int mt = F / (g.D / 16), ks = F - mt * (g.D / 16);
    o.r = 16 * mt + a;
    o.c = 16 * ks + b;
  } else {
    const int mc = F / (g.W / 16), kt = F - mc * (g.W / 16);
    o.c = 16 * mc + a;
    o.r = 16 * kt + b;
  }
  return o;
}

// Position of key channel c inside the key min / key scale arrays of a 2-bit slot: lane t of
// channel step ks reads channels (16 ks + 2t, +1, +8, +9) -- its B-fragment channels -- as one
// 16-byte vector.
QE_HD int kparam_pos(int c) { return (c & ~15) + (((c & 7) >> 1) << 2) + (c & 1) + (((c >> 3) & 1) << 1); }
// Position of token r inside the value min / value scale arrays: lane group gg = r % 8 reads its
// rows (16 mt + gg and 16 mt + gg + 8 for every token tile mt) as one vector.
QE_HD int vparam_pos(const Geo& g, int r) {
  return (r & 7) * (2 * (g.W / 16)) + (r >> 4) * 2 + ((r >> 3) & 1);
}

// ---------------------------------------------------------------------------- cache state
// Per-layer dynamic state, resident on the device and updated by the kernels themselves, so
// that every launch has step-invariant arguments (a decode step can be captured once in a CUDA
// graph and replayed).  All sequences of a layer share these counts.
struct LayerDev {
  int L;             // tokens per sequence
  int routed_upto;   // windows [0, routed_upto) have entered the candidate pool
  int n_full;        // Full windows per unit
  int n_quant;       // Quantized windows per unit
  int kf, kq;        // capacities at the last routing event
  unsigned done;     // blocks finished in the kernel that updates this header (last one commits)
  int pad;
};

// Capacity rule (see qe.h)
struct CapCfg {
  int mode, kf, kq;
  double frac_bf16, frac_int2, budget_frac;
};

// Arrays are indexed by the global unit gu = layer * units + (b * n_kv_heads + kvh).
struct State {
  int units;          // per layer
  int n_layers;
  int maxw;           // windows per sequence
  int capb, capq, caps;
  int n_sink, n_recent, G, Hq, Hkv;
  Geo geo;
  uint8_t* tier;      // [GU][maxw]
  int* bslot;         // [GU][maxw]
  int* qslot;         // [GU][maxw]
  int* sent;          // [GU][maxw] host store / ledger entry
  float* score;       // [GU][maxw]
  int2* blist;        // [GU][capb] {window, slot}; entry 0 is the sink {-1, 0}
  int2* qlist;        // [GU][capq]
  // Free bf16 and 2-bit slots, next to hand out first: entries [bfree_head, bfree_top) and
  // [0, qfree_top).  A slot freed by a demotion (bf16) or a promotion (2-bit) still holds that
  // window's exact data (bvictim / qvictim name the window, bprev / qprev the window's last
  // slot): it goes to the back, so it is handed out late, and the window takes it back without a
  // host transfer if nobody has taken it meanwhile.  Slots of evicted windows go to the front.
  int* bfree; int* bfree_head; int* bfree_top;   // [GU][capb], [GU], [GU]
  int* qfree; int* qfree_top;                    // [GU][capq], [GU]
  int* sfree; int* sfree_top;                    // [GU][caps], [GU] (store entries, a stack)
  int* bvictim;       // [GU][capb] window whose exact bf16 the slot holds, -1 if none
  int* qvictim;       // [GU][capq] window whose 2-bit codes the slot holds, -1 if none
  int* bprev;         // [GU][maxw] last bf16 slot of the window, -1 if none
  int* qprev;         // [GU][maxw] last 2-bit slot of the window, -1 if none
  uint8_t* bslab;     // [GU][capb][bslot_bytes]
  uint8_t* qslab;     // [GU][capq][qslot_bytes]
  int* qrange;        // [GU][capq] magnitudes of the parameters a 2-bit slot holds (qrange_word)
  uint8_t* hstore;    // device pointer to pinned host [GU][caps][bslot_bytes]
  uint8_t* hledger;   // device pointer to pinned host [GU][caps][qslot_bytes]
  unsigned* err;      // sticky flag
  unsigned long long* stats;  // [layers][N_STATS]
  LayerDev* ldev;     // [layers]
  CapCfg cap;
  int max_context;
};

// Capacity rule in double precision, operations in the order qe.h states, each rounded once
// (no fused multiply-add), so host, device and the reference give identical window counts.
QE_HD int qslot_bytes_of(int W, int D) { return 2 * (W * D / 4) + 8 * D + 8 * W; }
#if defined(__CUDA_ARCH__)
#define QE_DMUL(a, b) __dmul_rn((a), (b))
#define QE_DSUB(a, b) __dsub_rn((a), (b))
#define QE_DDIV(a, b) __ddiv_rn((a), (b))
#else
#define QE_DMUL(a, b) ((a) * (b))
#define QE_DSUB(a, b) ((a) - (b))
#define QE_DDIV(a, b) ((a) / (b))
#endif
QE_HD void capacities_at(const CapCfg& c, int n_sink, int n_recent, int W, int D, int L, int& kf, int& kq) {
  if (c.mode == 0) {
    kf = c.kf;
    kq = c.kq;
    return;
  }
  const double f = floor(QE_DDIV(QE_DSUB(QE_DSUB(QE_DMUL(c.frac_bf16, (double)L), (double)n_sink), (double)n_recent),
                                 (double)W));
  kf = f < 0 ? 0 : (int)f;
  double q;
  if (c.mode == 1) q = floor(QE_DDIV(QE_DMUL(c.frac_int2, (double)L), (double)W));
  else
    q = floor(QE_DDIV(QE_DMUL(QE_DMUL(QE_DSUB(c.budget_frac, c.frac_bf16), (double)L), 4.0 * D),
                      (double)qslot_bytes_of(W, D)));
  kq = q < 0 ? 0 : (int)q;
}

// Derived counts of one layer (identical on every thread that reads the same header).
struct LayerView {
  int L, nwin, nbw, nq;
};
QE_HD LayerView layer_view(const Geo& g, const LayerDev& h) {
  LayerView v;
  v.L = h.L;
  v.nwin = (h.L + g.W - 1) / g.W;
  v.nbw = 1 + h.n_full + (v.nwin - h.routed_upto);   // sink + Full + Pinned windows
  v.nq = h.n_quant;
  return v;
}

// ---------------------------------------------------------------------------- PTX helpers
#if defined(__CUDACC__)
__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (L2 only), its commit group, and the waits
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_but_newest() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// programmatic dependent launch: let the next launch on the stream begin / wait for the
// previous launch's completion and memory flush
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done != 0;
}
// the same test, allowed to suspend the thread until the phase completes (at most about ns
// nanoseconds): a waiting warp takes no issue slots from the working ones
__device__ __forceinline__ bool mbar_try_wait_sleep(unsigned bar, unsigned parity, unsigned ns) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(bar), "r"(parity), "r"(ns) : "memory");
  return done != 0;
}
__device__ __forceinline__ void bulk_g2s(unsigned dst, const void* src, unsigned bytes, unsigned bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// The same copy with an L2 policy: a stream read once per step (K/V tiles; the whole cache is
// many times the L2) is marked evict-first, so it does not push out what is reused (the layer's
// lists and partials, the queries, the code).
__device__ __forceinline__ unsigned long long l2_evict_first_policy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(unsigned dst, const void* src, unsigned bytes, unsigned bar,
                                              unsigned long long pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}
// 16-byte read-only load with an L2 policy (data that does not change during the kernel)
__device__ __forceinline__ uint4 ldg_hint(const void* p, unsigned long long pol) {
  uint4 v;
  asm("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
  return v;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                         unsigned b0, unsigned b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned movmatrix_t(unsigned a) {
  unsigned d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
// Register R (0..7) of a code word as an f16 pair (1 + code / 4): its codes sit at bits 2R and
// 2R + 16; the shift brings them to bits 8 and 24, the f16 mantissa's top two bits under the
// exponent of 1.0.
template <int R>
__device__ __forceinline__ unsigned code_pair_f16(unsigned w) {
  constexpr int SH = 8 - 2 * R;
  const unsigned x = SH >= 0 ? (w << (SH >= 0 ? SH : 0)) : (w >> (SH < 0 ? -SH : 0));
  unsigned d;
  asm("lop3.b32 %0, %1, 0x03000300, 0x3C003C00, 0xEA;" : "=r"(d) : "r"(x));   // (a & b) | c
  return d;
}
// the 4 f16x2 A-fragment registers of fragment F (0 or 1) of a code word
template <int F>
__device__ __forceinline__ void unpack_half(unsigned w, unsigned (&a)[4]) {
  a[0] = code_pair_f16<4 * F + 0>(w);
  a[1] = code_pair_f16<4 * F + 1>(w);
  a[2] = code_pair_f16<4 * F + 2>(w);
  a[3] = code_pair_f16<4 * F + 3>(w);
}
// The same pair as bf16 (1 + code / 4 is exact in bf16 too): the codes go to bits 5 and 21, the
// top two bits of the bf16 mantissa under the exponent of 1.0.
template <int R>
__device__ __forceinline__ unsigned code_pair_bf16(unsigned w) {
  constexpr int SH = 5 - 2 * R;
  const unsigned x = SH >= 0 ? (w << (SH >= 0 ? SH : 0)) : (w >> (SH < 0 ? -SH : 0));
  unsigned d;
  asm("lop3.b32 %0, %1, 0x00600060, 0x3F803F80, 0xEA;" : "=r"(d) : "r"(x));   // (a & b) | c
  return d;
}
template <int F>
__device__ __forceinline__ void unpack_half_bf16(unsigned w, unsigned (&a)[4]) {
  a[0] = code_pair_bf16<4 * F + 0>(w);
  a[1] = code_pair_bf16<4 * F + 1>(w);
  a[2] = code_pair_bf16<4 * F + 2>(w);
  a[3] = code_pair_bf16<4 * F + 3>(w);
}
#endif

// Range record of a 2-bit slot's parameters (written whenever a slot receives codes): the
// biased float32 exponents of the largest key scale (bits 0-7), of the largest value scale
// (bits 8-15) and of the smallest nonzero value scale (bits 16-23; 255 when every value scale
// is 0).  Scales are >= 0, so their bit patterns order like their values.
QE_HD int qrange_word(unsigned kscale_max_bits, unsigned vscale_max_bits, unsigned vscale_min_nonzero_bits) {
  const unsigned vmin = vscale_min_nonzero_bits == 0xFFFFFFFFu ? 255u : (vscale_min_nonzero_bits >> 23) & 0xFFu;
  return (int)(((kscale_max_bits >> 23) & 0xFFu) | (((vscale_max_bits >> 23) & 0xFFu) << 8) | (vmin << 16));
}
// Whether a 2-bit tile needs bf16 operands instead of f16 ones.  Its products meet the tensor
// cores as f16 truncated + remainder pairs: q_c s_c for the keys and 4 p s_V for the values,
// with p <= 2^8 (the softmax reference maximum is raised once a tile's scores pass it by 2^8).
// f16 holds them while |q| s_K < 2^15 and s_V < 2^5 (then 4 p s_V < 2^15); below s_V = 2^-13
// the remainder part falls into f16 subnormals and the value products lose relative precision.
// q_exp: the largest biased exponent of the unit's queries (bf16 and float32 share the bias).
QE_HD bool qrange_values_wide(int word) {
  const int evmax = (word >> 8) & 0xFF, evmin = (word >> 16) & 0xFF;
  return evmax >= 127 + 5 || evmin <= 127 - 14;
}
QE_HD bool qrange_wide(int word, int q_exp) {
  const int ek = word & 0xFF;
  return (ek > 0 && ek + q_exp >= 2 * 127 + 14) || qrange_values_wide(word);
}
#if defined(__CUDACC__)
__device__ __forceinline__ void mma_f16(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                        unsigned b0, unsigned b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// m16n8k8 with tf32 operands (float32 bit patterns whose 13 low mantissa bits are zero):
// A rows g, g + 8 at k = t (a0, a1) and k = t + 4 (a2, a3); B rows k = t (b0), t + 4 (b1) of
// column g; the accumulator layout is the m16n8k16 one
__device__ __forceinline__ void mma_tf32(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                         unsigned b0, unsigned b1) {
  asm(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// bf16x2 with round-toward-zero: lo -> low half
__device__ __forceinline__ unsigned pack_bf16x2_rz(float lo, float hi) {
  unsigned d;
  asm("cvt.rz.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// packed fp32 pair arithmetic (one instruction for two lanes' worth of values)
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  return (unsigned long long)__float_as_uint(a) | ((unsigned long long)__float_as_uint(b) << 32);
}
__device__ __forceinline__ float f2_lo(unsigned long long x) { return __uint_as_float((unsigned)x); }
__device__ __forceinline__ float f2_hi(unsigned long long x) { return __uint_as_float((unsigned)(x >> 32)); }
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// f16x2 with round-toward-zero: lo -> low half
__device__ __forceinline__ unsigned pack_f16x2_rz(float lo, float hi) {
  unsigned d;
  asm("cvt.rz.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// bf16x2 from two floats: lo -> low half, hi -> high half (round to nearest even)
__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
  unsigned d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf16lo_to_f32(unsigned x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi_to_f32(unsigned x) { return __uint_as_float(x & 0xFFFF0000u); }
#endif

}  // namespace qe
