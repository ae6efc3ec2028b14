// qe_verify.cu -- speculative verify of n_q drafts with one read of the cache (window tiering).
//
// H2O page, §5 (speculative decoding): each draft query attends over the cache and the drafts
// before it, and its window masses are held back until the drafts are accepted or rejected.
// The n_q draft queries of a unit share every cached key and value, so their attention is one
// dense contraction of (n_q x G) query rows against each window: this file runs it on the 5th-
// generation tensor cores (tcgen05.mma, accumulators in tensor memory), reading every window
// once for all rows, instead of one decode step per draft.
//
// Layout of the work: one CTA of 128 threads per (unit, split of the unit's windows).
//  * Rows: row r = j G + h is draft j's query head h (r < 64 = 16 drafts x 4 heads).  The mma
//    is M = 64; its accumulator row r sits in tensor-memory lane 32 (r / 16) + r % 16, so warp
//    w's lanes 0..15 own rows 16 w .. 16 w + 15 and each such thread runs its row's softmax.
//  * Per window (W tokens), all in shared memory in the no-swizzle K-major core-matrix layout
//    (8 rows x 16 bytes per core matrix, the two halves of a 16-wide K step 128 bytes apart):
//      - keys as the B operand of S = Q K^T: bf16 windows as stored; a 2-bit window's keys
//        dequantized (code * s + z, one float32 fma, as the oracle does) and split into three
//        bf16 parts (truncated, truncated remainder, rest: exact together), placed as three
//        blocks of W rows so that one mma chain over N = 3W gives all three partial products;
//      - values as the B operand of O += P V, channels as rows: bf16 values, or a 2-bit window's
//        codes as 1 + code / 4 (exact in bf16), the value scale folded into P and the offset
//        sum_t p_t (z_t - 4 s_t) kept per row in a register;
//      - P (times 4 s_V for 2-bit windows) as the A operand of O += P V, three exact bf16 parts
//        along K.
//    Q (bf16, exact) is loaded once.  Every operand is bf16, so all products are exact and
//    accumulate in float32: no magnitude leaves the operand format.
//  * S (up to 3W columns) and O (D columns) live in tensor memory; a row's online softmax rescales
//    its O row there (tcgen05.ld / st) when its reference maximum grows by more than 2^8.
//  * Causality among the drafts: draft j sees positions < L0 + j + 1.
//  * Per window and row the kernel writes the log2-sum-exp of the window's logits; the combine
//    kernel turns them into each draft's window masses once the row's normaliser is known.
// Waits are bounded (0.2 s); an expired wait sets the sticky timeout bit and the CTA leaves
// after the tensor-core work it issued has finished.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qe_kernels.cuh"

namespace qe {

constexpr int VF_THREADS = 256;   // warps 0-3 own the rows; all eight build the operands
constexpr int VF_ROWS = 64;
constexpr unsigned long long VF_WAIT_NS = 200000000ull;

template <int D, int W>
struct VfShape {
  static constexpr int NKQ = 3 * W;                       // key rows of S's B operand (3 parts)
  static constexpr int KP = 3 * W;                        // K extent of P (3 parts)
  static constexpr int SQ = VF_ROWS * D * 2;
  static constexpr int SBK = NKQ * D * 2;
  static constexpr int SBV = D * W * 2;
  static constexpr int SAP = VF_ROWS * KP * 2;
  static constexpr int BSLOT = 4 * W * D;
  static constexpr int QSLOT = 2 * (W * D / 4) + 8 * D + 8 * W;
  static constexpr int STAGE = ((BSLOT > QSLOT ? BSLOT : QSLOT) + 127) / 128 * 128;
  static constexpr int SMEM = SQ + SBK + SBV + SAP + 2 * STAGE;
  static constexpr int TO_OFF = NKQ <= 128 ? 128 : 256;  // tensor-memory column of O
  static constexpr int TMEM_COLS = TO_OFF + D <= 256 ? 256 : 512;
  // Dynamic shared memory requested per CTA: at least enough that no more CTAs share an SM than
  // its 512 tensor-memory columns hold (two of 256 columns, or one of 512).
  static constexpr int SMEM_FLOOR = TMEM_COLS == 256 ? 80 * 1024 : 120 * 1024;
  static constexpr int SMEM_REQ = SMEM > SMEM_FLOOR ? SMEM : SMEM_FLOOR;
};

// byte offset of element (row, k) of an operand with kdim elements per row, K-major, no swizzle
__device__ __forceinline__ int vf_canon(int row, int k, int kdim) {
  return (row >> 3) * (kdim >> 3) * 128 + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

// shared-memory matrix descriptor: start, leading byte offset (between the K halves of a core
// matrix pair, 128), stride byte offset (between 8-row groups), descriptor version 1, no swizzle
__device__ __forceinline__ unsigned long long vf_desc(const void* smem, unsigned sbo) {
  unsigned long long d = 0;
  d |= (unsigned long long)((smem_u32(smem) >> 4) & 0x3FFF);
  d |= (unsigned long long)((128u >> 4) & 0x3FFF) << 16;
  d |= (unsigned long long)((sbo >> 4) & 0x3FFF) << 32;
  d |= 1ull << 46;
  return d;
}

// instruction descriptor of kind::f16: bf16 A and B (K-major), float32 accumulator, M x N
__device__ __forceinline__ unsigned vf_idesc(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((unsigned)(n >> 3) << 17) | ((unsigned)(m >> 4) << 24);
}

__device__ __forceinline__ void vf_mma(unsigned tmem_d, unsigned long long a, unsigned long long b, unsigned idesc,
                                       bool accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}
__device__ __forceinline__ void vf_commit(unsigned bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void vf_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void vf_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void vf_proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive float32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void vf_ld16(unsigned taddr, float (&v)[16]) {
  unsigned r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void vf_st16(unsigned taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

// bounded wait on an mbarrier phase; false (and the timeout bit) when it expires
__device__ __forceinline__ bool vf_wait(unsigned bar, unsigned parity, unsigned* err) {
  unsigned long long t0 = 0;
  int spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if (++spins == 64) {
      spins = 0;
      const unsigned long long now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > VF_WAIT_NS) {
        atomicOr(err, ERR_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// the three bf16 parts of x (truncated, truncated remainder, rest), exact together
__device__ __forceinline__ void vf_split3(float x, unsigned& h, unsigned& m, unsigned& l) {
  const unsigned hb = __float_as_uint(x) & 0xFFFF0000u;
  const float r = x - __uint_as_float(hb);
  const unsigned mb = __float_as_uint(r) & 0xFFFF0000u;
  h = hb >> 16;
  m = mb >> 16;
  l = pack_bf16x2_rz(r - __uint_as_float(mb), 0.f) & 0xFFFFu;
}

// the same for a pair (x0, x1): three bf16x2 words, x0 in the low halves
__device__ __forceinline__ void vf_split3_pair(float x0, float x1, unsigned& h, unsigned& m, unsigned& l) {
  const unsigned h0 = __float_as_uint(x0) & 0xFFFF0000u, h1 = __float_as_uint(x1) & 0xFFFF0000u;
  const float r0 = x0 - __uint_as_float(h0), r1 = x1 - __uint_as_float(h1);
  const unsigned m0 = __float_as_uint(r0) & 0xFFFF0000u, m1 = __float_as_uint(r1) & 0xFFFF0000u;
  h = __byte_perm(h0, h1, 0x7632);
  m = __byte_perm(m0, m1, 0x7632);
  l = pack_bf16x2_rz(r0 - __uint_as_float(m0), r1 - __uint_as_float(m1));
}

template <int D, int W>
__global__ void __launch_bounds__(VF_THREADS) qe_verify_attn_kernel(const VerifyParams p) {
  using S = VfShape<D, W>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sBK = sQ + S::SQ;
  uint8_t* sBV = sBK + S::SBK;
  uint8_t* sAP = sBV + S::SBV;
  uint8_t* stg_base = sAP + S::SAP;
  __shared__ __align__(8) unsigned long long bar_stage[2], bar_s, bar_o;
  __shared__ unsigned s_tmem;
  __shared__ float s_vs[W], s_vz[W];   // 2-bit window: 4 s_V and z_V - 4 s_V per token
  __shared__ int s_stop;

  const State& st = p.st;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.x, split = blockIdx.y;
  const long long gu = (long long)p.layer * st.units + u;
  const int G = st.G;
  const Geo g{D, W};
  const LayerDev hd = st.ldev[p.layer];
  const LayerView lv = layer_view(g, hd);
  const int L = lv.L, nbw = lv.nbw, nq = lv.nq;
  const int b0 = (int)((long long)split * nbw / p.splits), b1 = (int)((long long)(split + 1) * nbw / p.splits);
  const int q0 = (int)((long long)split * nq / p.splits), q1 = (int)((long long)(split + 1) * nq / p.splits);
  const int nchunk = (b1 - b0) + (q1 - q0);
  const bool row_warp = warp < 4;                      // warps whose lanes 0..15 own the rows
  const int r = (warp & 3) * 16 + (lane & 15);         // the row this thread serves
  const bool row_valid = row_warp && lane < 16 && r < p.R;
  const int jdraft = r / G;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(S::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar_stage[0]), 1);
    mbar_init(smem_u32(&bar_stage[1]), 1);
    mbar_init(smem_u32(&bar_s), 1);
    mbar_init(smem_u32(&bar_o), 1);
    mbar_fence_init();
    s_stop = 0;
  }
  // Q rows (zero beyond R) and zero P rows beyond R, once
  {
    const int b = u / st.Hkv, kvh = u - b * st.Hkv, B = st.units / st.Hkv;
    for (int i = tid; i < VF_ROWS * (D / 2); i += VF_THREADS) {
      const int rr = i / (D / 2), c = 2 * (i - rr * (D / 2));
      unsigned val = 0u;
      if (rr < p.R) {
        const int jj = rr / G, hh = rr - jj * G;
        val = *reinterpret_cast<const unsigned*>(p.q + (((size_t)jj * B + b) * st.Hq + kvh * G + hh) * D + c);
      }
      *reinterpret_cast<unsigned*>(sQ + vf_canon(rr, c, D)) = val;
    }
    for (int i = tid; i < VF_ROWS * (S::KP / 2); i += VF_THREADS) {
      const int rr = i / (S::KP / 2), k = 2 * (i - rr * (S::KP / 2));
      if (rr >= p.R) *reinterpret_cast<unsigned*>(sAP + vf_canon(rr, k, S::KP)) = 0u;
    }
  }
  vf_proxy_fence();
  vf_fence_before();
  __syncthreads();
  vf_fence_after();
  const unsigned tS = s_tmem, tO = s_tmem + S::TO_OFF;
  const unsigned lane_off = (unsigned)((warp & 3) * 32) << 16;

  // chunk c: bf16 entry b0 + c, then 2-bit entry q0 + (c - (b1 - b0))
  auto chunk_entry = [&](int c, bool& is_q, int& eidx) -> int2 {
    if (c < b1 - b0) {
      is_q = false;
      eidx = b0 + c;
      return st.blist[gu * st.capb + eidx];
    }
    is_q = true;
    const int qi = q0 + (c - (b1 - b0));
    eidx = nbw + qi;
    return st.qlist[gu * st.capq + qi];
  };
  int pending[2] = {-1, -1};   // thread 0: chunk whose copy a stage has in flight, or -1
  auto issue = [&](int c, int s) {
    if (tid != 0 || c >= nchunk) return;
    bool is_q;
    int eidx;
    const int2 e = chunk_entry(c, is_q, eidx);
    const unsigned bar = smem_u32(&bar_stage[s]);
    const uint8_t* src;
    unsigned bytes;
    if (!is_q) {
      if (e.y < 0 || e.y >= st.capb) { atomicOr(st.err, ERR_TABLE); s_stop = 1; return; }
      src = st.bslab + (gu * st.capb + e.y) * (long long)S::BSLOT;
      bytes = S::BSLOT;
    } else {
      if (e.y < 0 || e.y >= st.capq) { atomicOr(st.err, ERR_TABLE); s_stop = 1; return; }
      src = st.qslab + (gu * st.capq + e.y) * (long long)S::QSLOT;
      bytes = S::QSLOT;
    }
    mbar_expect_tx(bar, bytes);
    bulk_g2s(smem_u32(stg_base + (size_t)s * S::STAGE), src, bytes, bar);
    pending[s] = c;
  };
  issue(0, 0);
  issue(1, 1);

  float mref = -INFINITY, lsum = 0.f, zs = 0.f;
  bool o_init = false;
  bool s_left = false;   // an S mma whose completion was not seen
  int c = 0;
  bool ok = true;
  for (; c < nchunk; ++c) {
    const int sidx = c & 1;
    bool is_q;
    int eidx;
    const int2 ent = chunk_entry(c, is_q, eidx);
    const int win = ent.x;
    // previous P V done (its operands and O may be rewritten) and this chunk's copy landed; every
    // thread agrees on the outcome before anyone leaves the loop
    bool w_ok = c == 0 || vf_wait(smem_u32(&bar_o), (c - 1) & 1, st.err);
    w_ok = vf_wait(smem_u32(&bar_stage[sidx]), (c >> 1) & 1, st.err) && w_ok;
    if (tid == 0 && w_ok) pending[sidx] = -1;
    if (!__syncthreads_and(w_ok) || s_stop) { ok = false; break; }
    const uint8_t* sp = stg_base + (size_t)sidx * S::STAGE;
    // ---- operands.  Layout arithmetic at compile time (every divisor is a power of two); in the
    // K-major core-matrix layout, row + 8 is the next 8-row group (+ kdim * 16 bytes) and column
    // + 8 the next core matrix (+ 128 bytes), so each piece's four registers land at one base plus
    // constants.
    if (!is_q) {
      // a bf16 slot in mma fragment order: each 16-byte piece is one lane's four registers of a
      // 16 x 16 fragment (rows g, g + 8 at columns 2t, 2t + 8); keys have tokens as rows, values
      // channels as rows
      constexpr int KS = D / 16, SUBB = 64 * D, NKC = (W / 16) * KS * 32;
      for (int i = tid; i < 2 * NKC; i += VF_THREADS) {
        const bool value = i >= NKC;
        const int ii = value ? i - NKC : i;
        const int ln = ii & 31, blk = (ii >> 5) % KS, sub = (ii >> 5) / KS;
        const int gg = ln >> 2, tt = ln & 3;
        const uint4 x = *reinterpret_cast<const uint4*>(sp + sub * SUBB + (value ? 32 * D : 0) + blk * 512 + ln * 16);
        // keys: token 16 sub + gg, channel 16 blk + 2 tt; values: channel 16 blk + gg, token 16 sub + 2 tt
        uint8_t* dst = value ? sBV + vf_canon(16 * blk + gg, 16 * sub + 2 * tt, W)
                             : sBK + vf_canon(16 * sub + gg, 16 * blk + 2 * tt, D);
        const int row8 = value ? W * 16 : D * 16;   // + 8 rows
        *reinterpret_cast<unsigned*>(dst) = x.x;
        *reinterpret_cast<unsigned*>(dst + row8) = x.y;
        *reinterpret_cast<unsigned*>(dst + 128) = x.z;
        *reinterpret_cast<unsigned*>(dst + row8 + 128) = x.w;
      }
    } else {
      // 2-bit codes: word wi of a code block holds fragments 2 wj, 2 wj + 1 of one lane (wj and
      // the lane from wi), register reg of fragment f at bits 8 f + 2 reg (+ 16 for the second
      // element); fragment 2 wj + 1 is the next 16-wide K step (keys) or token step (values)
      constexpr int KS = D / 16, KT = W / 16, WPL = KT * KS / 2, CW = WPL < 4 ? WPL : 4, NWORD = 32 * WPL;
      const float* kmin = reinterpret_cast<const float*>(sp + g.off_kmin());
      const float* kscale = reinterpret_cast<const float*>(sp + g.off_kscale());
      static_assert(KS % 2 == 0, "a key word's two fragments are consecutive channel steps");
      for (int i = tid; i < 2 * NWORD; i += VF_THREADS) {
        const bool value = i >= NWORD;
        const int wi = value ? i - NWORD : i;
        const unsigned w = *reinterpret_cast<const unsigned*>(sp + (value ? g.off_vcode() : 0) + 4 * wi);
        const int chunk = wi / (32 * CW), rem = wi % (32 * CW);
        const int ln = rem / CW, wj = chunk * CW + rem % CW;
        const int gg = ln >> 2, tt = ln & 3;
        const int F0 = 2 * wj;
        if (!value) {
          const int mt = F0 / KS, ks = F0 % KS;   // fragment 2 wj + 1: channel step ks + 1
          const int t = 16 * mt + gg, ch = 16 * ks + 2 * tt;
          uint8_t* dst = sBK + vf_canon(t, ch, D);
#pragma unroll
          for (int f = 0; f < 2; ++f)
#pragma unroll
            for (int reg = 0; reg < 4; ++reg) {
              const int c2 = ch + 16 * f + 8 * (reg >> 1);
              const float2 sc = *reinterpret_cast<const float2*>(kscale + kparam_pos(c2));
              const float2 mn = *reinterpret_cast<const float2*>(kmin + kparam_pos(c2));
              const unsigned x = w >> (8 * f + 2 * reg);
              unsigned hp, mp, lp;
              vf_split3_pair(fmaf((float)(x & 3u), sc.x, mn.x), fmaf((float)((x >> 16) & 3u), sc.y, mn.y), hp, mp,
                             lp);
              uint8_t* d0 = dst + f * 256 + (reg & 1) * (D * 16) + (reg >> 1) * 128;
              *reinterpret_cast<unsigned*>(d0) = hp;
              *reinterpret_cast<unsigned*>(d0 + W * D * 2) = mp;        // part 2: rows W ..
              *reinterpret_cast<unsigned*>(d0 + 2 * W * D * 2) = lp;    // part 3: rows 2W ..
            }
        } else {
          // fragment 2 wj + 1: token step kt + 1, or with one token step (W = 16) the next channel
          // block (16 rows further)
          const int mc = F0 / KT, kt = F0 % KT;
          constexpr int F1 = KT >= 2 ? 256 : 2 * W * 16;
          uint8_t* dst = sBV + vf_canon(16 * mc + gg, 16 * kt + 2 * tt, W);
#pragma unroll
          for (int f = 0; f < 2; ++f)
#pragma unroll
            for (int reg = 0; reg < 4; ++reg) {
              const unsigned x = w >> (8 * f + 2 * reg);
              *reinterpret_cast<unsigned*>(dst + f * F1 + (reg & 1) * (W * 16) + (reg >> 1) * 128) =
                  0x3F803F80u | ((x & 3u) << 5) | (((x >> 16) & 3u) << 21);
            }
        }
      }
      if (tid < W) {
        const float vsc = reinterpret_cast<const float*>(sp + g.off_vscale())[vparam_pos(g, tid)];
        const float vmn = reinterpret_cast<const float*>(sp + g.off_vmin())[vparam_pos(g, tid)];
        s_vs[tid] = 4.f * vsc;
        s_vz[tid] = vmn - 4.f * vsc;
      }
    }
    vf_proxy_fence();
    vf_fence_before();
    __syncthreads();
    vf_fence_after();
    issue(c + 2, sidx);   // every thread has read the stage
    // ---- S = Q K^T (N = W, or 3W for a 2-bit window's three key parts)
    const int nk = is_q ? 3 * W : W;
    if (tid == 0) {
      const unsigned idesc = vf_idesc(VF_ROWS, nk);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        vf_mma(tS, vf_desc(sQ + ks * 256, (D / 8) * 128), vf_desc(sBK + ks * 256, (D / 8) * 128), idesc, ks > 0);
      vf_commit(smem_u32(&bar_s));
    }
    if (!__syncthreads_and(vf_wait(smem_u32(&bar_s), c & 1, st.err))) {
      ok = false;
      ++c;   // this chunk's S mma was issued: its completion is awaited below with the P V ones
      s_left = true;
      break;
    }
    vf_fence_after();
    // ---- softmax of this window, per row
    if (row_warp) {   // warps 0-3: the sub-partitions holding the rows
      int lo, hi, pos0;
      if (!is_q && win < 0) {
        lo = 0;
        hi = st.n_sink < L ? st.n_sink : L;
        pos0 = 0;
      } else {
        lo = win == 0 ? st.n_sink : 0;
        hi = is_q ? W : (L - win * W < W ? L - win * W : W);
        pos0 = win * W;
      }
      // valid tokens of the window for this row: [tmin, tmax); draft j sees positions < L0 + j + 1
      const int tmin = lo, tmax = min(hi, p.L0 + jdraft + 1 - pos0);
      float x[W];
#pragma unroll
      for (int t0 = 0; t0 < W; t0 += 16) {
        float a[16];
        vf_ld16(tS + lane_off + t0, a);
        if (is_q) {
          float b[16], d[16];
          vf_ld16(tS + lane_off + W + t0, b);
          vf_ld16(tS + lane_off + 2 * W + t0, d);
#pragma unroll
          for (int i = 0; i < 16; ++i) a[i] = (a[i] + b[i]) + d[i];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) x[t0 + i] = a[i] * p.scale_log2;
      }
      if (tmin > 0 || tmax < W) {
#pragma unroll
        for (int t = 0; t < W; ++t)
          if (t < tmin || t >= tmax) x[t] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < W; ++t) mx = fmaxf(mx, x[t]);
      const bool raise = row_valid && mx > mref + 8.f;
      const float mnew = raise ? mx : mref;
      const float alpha = (raise && mref != -INFINITY) ? ex2(mref - mnew) : 1.f;
      if (__any_sync(0xffffffffu, raise && o_init && mref != -INFINITY)) {
        // rescale this warp's O rows (the warp's loads and stores are collective)
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          float o[16];
          vf_ld16(tO + lane_off + c0, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= alpha;
          vf_st16(tO + lane_off + c0, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      if (raise) {
        lsum *= alpha;
        zs *= alpha;
        mref = mnew;
      }
      const float muse = mref == -INFINITY ? 0.f : mref;
      float mass = 0.f, zadd = 0.f;
      if (row_valid) {
        uint8_t* prow = sAP + vf_canon(r, 0, S::KP);   // K index t: + (t / 8) 128 + (t % 8) 2 bytes
#pragma unroll
        for (int t = 0; t < W; t += 2) {
          float y[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = ex2(x[t + e] - muse);
            mass += pv;
            y[e] = pv;
            if (is_q) {
              zadd = fmaf(pv, s_vz[t + e], zadd);
              y[e] = pv * s_vs[t + e];
            }
          }
          unsigned hp, mp, lp;
          vf_split3_pair(y[0], y[1], hp, mp, lp);
          uint8_t* d0 = prow + (t >> 3) * 128 + (t & 7) * 2;
          *reinterpret_cast<unsigned*>(d0) = hp;
          *reinterpret_cast<unsigned*>(d0 + W * 16) = mp;       // K index W + t
          *reinterpret_cast<unsigned*>(d0 + 2 * W * 16) = lp;   // K index 2W + t
        }
        lsum += mass;
        zs += zadd;
        p.lse[((long long)u * p.ent_cap + eidx) * VF_ROWS + r] = mass > 0.f ? muse + lg2(mass) : -INFINITY;
      }
    }
    vf_proxy_fence();
    vf_fence_before();
    __syncthreads();
    vf_fence_after();
    // ---- O += P V: three parts of P along K, each against the same value block
    if (tid == 0) {
      const unsigned idesc = vf_idesc(VF_ROWS, D);
#pragma unroll
      for (int part = 0; part < 3; ++part)
#pragma unroll
        for (int kt = 0; kt < W / 16; ++kt)
          vf_mma(tO, vf_desc(sAP + (part * (W / 16) + kt) * 256, (S::KP / 8) * 128),
                 vf_desc(sBV + kt * 256, (W / 8) * 128), idesc, o_init || part > 0 || kt > 0);
      vf_commit(smem_u32(&bar_o));
    }
    o_init = true;
  }
  // Before tensor memory is read or freed, the tensor-core work issued must have finished (the
  // last P V: chunk c - 1 on a normal exit; after an expired wait also a pending S mma), and
  // before the CTA leaves, the copies still in flight must have landed (bounded waits).
  if (s_left) vf_wait(smem_u32(&bar_s), (c - 1) & 1, st.err);
  if (o_init) vf_wait(smem_u32(&bar_o), ((s_left ? c - 1 : c) - 1) & 1, st.err);
  if (tid == 0)
    for (int s = 0; s < 2; ++s)
      if (pending[s] >= 0) vf_wait(smem_u32(&bar_stage[s]), (pending[s] >> 1) & 1, st.err);
  vf_fence_after();
  const size_t pbase = ((size_t)u * p.splits + split) * VF_ROWS;
  if (ok && row_warp) {
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 16) {
      float o[16];
      if (o_init) vf_ld16(tO + lane_off + c0, o);
      else {
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = 0.f;
      }
      if (row_valid) {
        float* po = p.part_o + (pbase + r) * D + c0;
#pragma unroll
        for (int i = 0; i < 16; ++i) po[i] = o[i] + zs;
      }
    }
    if (row_valid) p.part_ml[pbase + r] = make_float2(mref, lsum);
  }
  vf_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(s_tmem), "r"(S::TMEM_COLS) : "memory");
}

// ------------------------------------------------------------------------------ combine
// One CTA per unit: merge each row's splits into draft j's output for head h, and turn every
// window's per-row log2-sum-exp into draft j's window mass (summed over its G heads), written
// to delta[j][unit][window] for qe_verify_commit.
constexpr int VF_COMBINE_THREADS = 256;
constexpr int VF_MAX_SPLITS = 16;

template <int D>
__global__ void __launch_bounds__(VF_COMBINE_THREADS) qe_verify_combine_kernel(const VerifyParams p, void* out,
                                                                              int out_fp32, float* delta,
                                                                              long long qstride) {
  const State& st = p.st;
  const int u = blockIdx.x, tid = threadIdx.x;
  const int G = st.G;
  const long long gu = (long long)p.layer * st.units + u;
  __shared__ float s_sc[VF_ROWS][VF_MAX_SPLITS];
  __shared__ float s_inv[VF_ROWS], s_lse[VF_ROWS];
  const Geo g{D, st.geo.W};
  const LayerView lv = layer_view(g, st.ldev[p.layer]);
  // row statistics
  if (tid < p.R) {
    const float2* ml = p.part_ml + (size_t)u * p.splits * VF_ROWS + tid;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, ml[(size_t)s * VF_ROWS].x);
    const float Mu = M == -INFINITY ? 0.f : M;
    float Ls = 0.f;
    for (int s = 0; s < p.splits; ++s) {
      const float2 v = ml[(size_t)s * VF_ROWS];
      const float sc = v.y > 0.f ? ex2(v.x - Mu) : 0.f;
      s_sc[tid][s] = sc;
      Ls = fmaf(v.y, sc, Ls);
    }
    s_inv[tid] = 1.f / Ls;
    s_lse[tid] = Mu + lg2(Ls);
  }
  __syncthreads();
  // outputs: draft j, head h, channel c
  const int b = u / st.Hkv, kvh = u - b * st.Hkv;
  for (int i = tid; i < p.R * D; i += VF_COMBINE_THREADS) {
    const int rr = i / D, c = i - rr * D;
    float acc = 0.f;
    for (int s = 0; s < p.splits; ++s)
      if (s_sc[rr][s] != 0.f) acc = fmaf(p.part_o[(((size_t)u * p.splits + s) * VF_ROWS + rr) * D + c], s_sc[rr][s], acc);
    const float o = acc * s_inv[rr];
    const int jj = rr / G, hh = rr - jj * G;
    const size_t oi = (((size_t)jj * st.units / st.Hkv + b) * st.Hq + kvh * G + hh) * D + c;
    if (out_fp32) reinterpret_cast<float*>(out)[oi] = o;
    else reinterpret_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(o);
  }
  // window masses per draft
  const int nent = lv.nbw + lv.nq;
  for (int i = tid; i < nent * p.n_q; i += VF_COMBINE_THREADS) {
    const int e = i / p.n_q, jj = i - e * p.n_q;
    const int2 ent = e < lv.nbw ? st.blist[gu * st.capb + e] : st.qlist[gu * st.capq + (e - lv.nbw)];
    if (ent.x < 0 || ent.x >= st.maxw) continue;   // the sink is not scored
    const float* ls = p.lse + ((long long)u * p.ent_cap + e) * VF_ROWS + jj * G;
    float dS = 0.f;
    for (int hh = 0; hh < G; ++hh) dS += ex2(ls[hh] - s_lse[jj * G + hh]);
    delta[jj * qstride + (long long)u * st.maxw + ent.x] = dS;
  }
}

// ------------------------------------------------------------------------------ launchers
template <int D, int W>
static cudaError_t vf_launch_t(const VerifyParams& p, void* out, int out_fp32, float* delta, long long qstride,
                               cudaStream_t s) {
  using S = VfShape<D, W>;
  qe_verify_attn_kernel<D, W><<<dim3(p.st.units, p.splits), VF_THREADS, S::SMEM_REQ, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  qe_verify_combine_kernel<D><<<p.st.units, VF_COMBINE_THREADS, 0, s>>>(p, out, out_fp32, delta, qstride);
  return cudaGetLastError();
}

template <int D, int W>
static cudaError_t vf_prepare_t() {
  return cudaFuncSetAttribute(qe_verify_attn_kernel<D, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              VfShape<D, W>::SMEM_REQ);
}

cudaError_t prepare_verify_kernels(int D, int W) {
  if (D == 128 && W == 16) return vf_prepare_t<128, 16>();
  if (D == 128 && W == 32) return vf_prepare_t<128, 32>();
  if (D == 128 && W == 64) return vf_prepare_t<128, 64>();
  if (D == 64 && W == 16) return vf_prepare_t<64, 16>();
  if (D == 64 && W == 32) return vf_prepare_t<64, 32>();
  if (D == 64 && W == 64) return vf_prepare_t<64, 64>();
  return cudaErrorInvalidValue;
}

cudaError_t launch_verify_fused(const VerifyParams& p, void* out, int out_fp32, float* delta, long long qstride,
                                cudaStream_t s) {
  const int D = p.st.geo.D, W = p.st.geo.W;
  if (p.splits < 1 || p.splits > VF_MAX_SPLITS || p.R < 1 || p.R > VF_ROWS) return cudaErrorInvalidValue;
  if (D == 128 && W == 16) return vf_launch_t<128, 16>(p, out, out_fp32, delta, qstride, s);
  if (D == 128 && W == 32) return vf_launch_t<128, 32>(p, out, out_fp32, delta, qstride, s);
  if (D == 128 && W == 64) return vf_launch_t<128, 64>(p, out, out_fp32, delta, qstride, s);
  if (D == 64 && W == 16) return vf_launch_t<64, 16>(p, out, out_fp32, delta, qstride, s);
  if (D == 64 && W == 32) return vf_launch_t<64, 32>(p, out, out_fp32, delta, qstride, s);
  if (D == 64 && W == 64) return vf_launch_t<64, 64>(p, out, out_fp32, delta, qstride, s);
  return cudaErrorInvalidValue;
}

int verify_max_rows() { return VF_ROWS; }
int verify_min_rows() { return 48; }
int verify_max_splits() { return VF_MAX_SPLITS; }

}  // namespace qe
