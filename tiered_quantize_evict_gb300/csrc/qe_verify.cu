// qe_verify.cu -- speculative verify of n_q drafts with one read of the cache (window tiering).
//
// H2O page, §5 (speculative decoding): each draft query attends over the cache and the drafts
// before it, and its window masses are held back until the drafts are accepted or rejected.
// The n_q draft queries of a unit share every cached key and value, so their attention is a
// dense contraction of the (n_q x G) query rows against each window: this file runs it on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory), reading every window
// once for all rows, instead of one decode step per draft.
//
// One CTA of 288 threads (9 warps) per (unit, split of the unit's windows); a window is a
// "chunk".
//  * Rows: row r = j G + h (draft j, query head h), r < 64.
//  * S = Q K^T per chunk: M = 64 rows, N = W tokens (bf16 window) or 3W (a 2-bit window's
//    keys dequantized as code * s + z, one float32 fma as the oracle does, and split into three
//    bf16 parts -- truncated, truncated remainder, rest -- that are exact together; the three
//    parts' products land in three column blocks and are summed in float32).  Q is bf16, so
//    every product is exact.  Accumulator row r sits in tensor-memory lane 32 (r / 16) + r % 16.
//  * O += P V per chunk: M = 64 rows (A: P), N = D channels (B: values with channels as rows),
//    K = the chunk's tokens, once for P's truncated bf16 part and once for its rounded
//    remainder (P to about 17 significant bits).  A 2-bit window's values enter as 1 + code / 4
//    (exact in bf16) with 4 s_V folded into P and sum_t p_t (z_t - 4 s_t) kept per row.  O
//    lives in tensor memory for the whole CTA, in the same lanes as S.
//  * Warps 0-3 run the softmax, warp w on rows 16 w .. 16 w + 15: the 16x256b tensor-memory
//    load gives lane T the rows 16 w + T / 4 and 16 w + 8 + T / 4 and two adjacent columns of
//    every 8-column block (the mma accumulator fragment), so a row's four lanes reduce with two
//    shuffles.  A row's reference maximum grows lazily (by more than 2^8 in the log2 domain)
//    and the warp rescales its own rows of O in tensor memory.
//  * Warps 4-7 build the operands of the next chunks (keys through per-warp tables of the three
//    bf16 parts of each channel's four codes; values; P is written by the softmax warps), in
//    the no-swizzle K-major core-matrix layout (8 rows x 16 bytes per core matrix, the two
//    halves of a 16-wide K step 128 bytes apart), through stmatrix.  Keys, values and P are
//    double-buffered; S is single-buffered (the softmax copies it to registers first).  2-bit
//    slots arrive by bulk copies three chunks ahead; bf16 slots by direct loads a chunk ahead.
//  * Warp 8 (one lane) issues the tensor-core work -- S of chunk c, then P V of chunk c - 1 --
//    and the stage refills.
//  * Causality among the drafts: draft j sees positions < L0 + j + 1.
//  * Per window and row the kernel writes the log2-sum-exp of the window's logits; the combine
//    kernel turns them into each draft's window masses once the row's normaliser is known.
// Handshakes (mbarriers): stage[s] (a 2-bit slot landed), stfree[s] (the builders are done
// with a stage), s (S complete), sfree (the softmax warps have read S), sk[b] (the S that read
// key buffer b is complete), keys[b] (keys of buffer b written), built[b] (values of buffer b
// written), p[b] (P of buffer b written, and any rescale of O done), o[b] (the P V of buffer b
// is complete).  Producers arrive once per warp after __syncwarp, or by tcgen05.commit.  Every
// wait is bounded (0.2 s); an expired wait sets the sticky timeout bit and an abort flag that
// ends every warp's loop, and the CTA leaves after the tensor-core work and copies it issued
// have finished.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "qe_kernels.cuh"

namespace qe {

constexpr int VF_THREADS = 288;   // warps 0-3: softmax; warps 4-7: operands; warp 8: tensor-core issue
constexpr int VF_ROWS = 64;
constexpr int VF_STAGES = 3;
constexpr unsigned long long VF_WAIT_NS = 200000000ull;

template <int D, int W>
struct VfShape {
  static constexpr int NKQ = 3 * W;                       // key rows of S's B operand (3 parts)
  static constexpr int KP = 2 * W;                        // K extent of P (2 parts)
  static constexpr int SQ = VF_ROWS * D * 2;
  static constexpr int SBK = NKQ * D * 2;
  static constexpr int SBV = D * W * 2;
  static constexpr int SAP = VF_ROWS * KP * 2;
  static constexpr int BSLOT = 4 * W * D;
  static constexpr int QSLOT = 2 * (W * D / 4) + 8 * D + 8 * W;
  static constexpr int STAGE = (QSLOT + 127) / 128 * 128;
  static constexpr int OFF_BK = SQ;
  static constexpr int OFF_BV = OFF_BK + 2 * SBK;
  static constexpr int OFF_AP = OFF_BV + 2 * SBV;
  static constexpr int OFF_STG = OFF_AP + 2 * SAP;
  static constexpr int OFF_TAB = OFF_STG + VF_STAGES * STAGE;   // key tables: 4 x [32 channels][4 codes] x 8 B
  static constexpr int SMEM = OFF_TAB + 4 * 1024;
  static constexpr int TO_OFF = (NKQ + 63) / 64 * 64;     // tensor memory: S at column 0, O (D columns) here
  static constexpr int TMEM_COLS = TO_OFF + D <= 256 ? 256 : 512;
  static constexpr bool FITS2 = 2 * (SMEM + 4096) <= 228 * 1024;   // two CTAs' shared memory per SM
  static constexpr int CTAS_PER_SM = TMEM_COLS == 256 && FITS2 ? 2 : 1;
  // Dynamic shared memory requested per CTA: at least enough that no more CTAs share an SM than
  // its 512 tensor-memory columns hold (two of 256 columns, or one of 512).
  static constexpr int SMEM_FLOOR = CTAS_PER_SM == 2 ? 80 * 1024 : 120 * 1024;
  static constexpr int SMEM_REQ = SMEM > SMEM_FLOOR ? SMEM : SMEM_FLOOR;
  static_assert(SMEM_REQ + 4096 <= 227 * 1024, "verify tile exceeds shared memory");
  static_assert(CTAS_PER_SM == 1 || 2 * (SMEM_REQ + 4096) <= 228 * 1024, "two CTAs must fit an SM");
};

// byte offset of element (row, k) of an operand with kdim elements per row, K-major, no swizzle
__device__ __forceinline__ int vf_canon(int row, int k, int kdim) {
  return (row >> 3) * (kdim >> 3) * 128 + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

// shared-memory matrix descriptor: start, leading byte offset (between the K halves of a core
// matrix pair, 128), stride byte offset (between 8-row groups), descriptor version 1, no swizzle
__device__ __forceinline__ unsigned long long vf_desc(unsigned saddr, unsigned sbo) {
  unsigned long long d = 0;
  d |= (unsigned long long)((saddr >> 4) & 0x3FFF);
  d |= (unsigned long long)((128u >> 4) & 0x3FFF) << 16;
  d |= (unsigned long long)((sbo >> 4) & 0x3FFF) << 32;
  d |= 1ull << 46;
  return d;
}

// instruction descriptor of kind::f16: bf16 A and B (K-major), float32 accumulator, M x N
__host__ __device__ constexpr unsigned vf_idesc(int m, int n) {
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
__device__ __forceinline__ void vf_arrive(unsigned bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// named barrier of one warp group (128 threads); the reductions return the group's AND / OR
__device__ __forceinline__ void vf_group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ bool vf_group_and(int id, bool v) {
  unsigned r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.and.pred p, %2, 128, q;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((unsigned)v), "r"(id)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ bool vf_group_or(int id, bool v) {
  unsigned r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.or.pred p, %2, 128, q;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((unsigned)v), "r"(id)
      : "memory");
  return r != 0;
}
// four 8 x 8 b16 matrices: register k of lane T is row T / 4, columns 2 (T % 4), +1 of matrix k;
// lane i gives the address of row i % 8 of matrix i / 8
__device__ __forceinline__ void vf_stmatrix4(unsigned saddr, unsigned r0, unsigned r1, unsigned r2, unsigned r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3)
               : "memory");
}

// Waits for this thread's tensor-memory loads; the registers pass through empty volatile asm
// statements after the wait, so that no use of them is scheduled before it.
template <int N>
__device__ __forceinline__ void vf_wait_ld(unsigned (&v)[N]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(v[i]));
}

// 16 consecutive float32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void vf_ld16(unsigned taddr, float (&v)[16]) {
  unsigned r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  vf_wait_ld(r);
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

// NB 8-column blocks of 16 lanes (16x256b shape): v[4 j + e] = (lane T / 4, column 8 j + 2 (T % 4)
// + e), v[4 j + 2 + e] = (lane 8 + T / 4, same column); the caller waits (tcgen05.wait::ld)
template <int NB>
__device__ __forceinline__ void vf_ld_rows(unsigned taddr, unsigned (&v)[4 * NB]);
template <>
__device__ __forceinline__ void vf_ld_rows<2>(unsigned taddr, unsigned (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}
template <>
__device__ __forceinline__ void vf_ld_rows<4>(unsigned taddr, unsigned (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
template <>
__device__ __forceinline__ void vf_ld_rows<8>(unsigned taddr, unsigned (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
// 4 8-column blocks (32 columns) of 16 lanes, the 16x256b layout of vf_ld_rows<4>
__device__ __forceinline__ void vf_st_rows4(unsigned taddr, const unsigned (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// One test of an mbarrier phase that may suspend the thread until the phase completes, for at
// most about 20 us: a waiting warp takes no issue slots from the working ones.
__device__ __forceinline__ bool vf_try_wait(unsigned bar, unsigned parity) {
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
// Bounded wait on an mbarrier phase.  False when it expires (the timeout bit and the abort flag
// are set) or when another thread has raised the abort flag meanwhile.
__device__ __forceinline__ bool vf_wait(unsigned bar, unsigned parity, unsigned* err, volatile int* abort_flag) {
  if (vf_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!vf_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > VF_WAIT_NS) {
      atomicOr(err, ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}
// the same without the abort flag: the exit path's wait for work already issued
__device__ __forceinline__ void vf_drain(unsigned bar, unsigned parity, unsigned* err) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > VF_WAIT_NS) {
      atomicOr(err, ERR_TIMEOUT);
      return;
    }
}

// the three bf16 parts of a pair (x0, x1) -- truncated, truncated remainder, rest (truncated),
// exact together -- as three bf16x2 words, x0 in the low halves
__device__ __forceinline__ void vf_split3_pair(float x0, float x1, unsigned& h, unsigned& m, unsigned& l) {
  const unsigned h0 = __float_as_uint(x0) & 0xFFFF0000u, h1 = __float_as_uint(x1) & 0xFFFF0000u;
  const float r0 = x0 - __uint_as_float(h0), r1 = x1 - __uint_as_float(h1);
  const unsigned m0 = __float_as_uint(r0) & 0xFFFF0000u, m1 = __float_as_uint(r1) & 0xFFFF0000u;
  h = __byte_perm(h0, h1, 0x7632);
  m = __byte_perm(m0, m1, 0x7632);
  l = pack_bf16x2_rz(r0 - __uint_as_float(m0), r1 - __uint_as_float(m1));
}
// two bf16 parts of a pair: truncated, and the remainder rounded to nearest
__device__ __forceinline__ void vf_split2_pair(float x0, float x1, unsigned& h, unsigned& l) {
  const unsigned h0 = __float_as_uint(x0) & 0xFFFF0000u, h1 = __float_as_uint(x1) & 0xFFFF0000u;
  h = __byte_perm(h0, h1, 0x7632);
  l = pack_bf16x2(x0 - __uint_as_float(h0), x1 - __uint_as_float(h1));
}
// a small integer code (0..3) as float32
__device__ __forceinline__ float vf_code_f(unsigned x) { return __uint_as_float(0x4B000000u | x) - 8388608.f; }

template <int D, int W>
__global__ void __launch_bounds__(VF_THREADS, VfShape<D, W>::CTAS_PER_SM) qe_verify_attn_kernel(const VerifyParams p) {
  using S = VfShape<D, W>;
  constexpr int KS = D / 16, KT = W / 16, NB = W / 8;
  constexpr int WPL = (W / 16) * (D / 16) / 2, CW = WPL < 4 ? WPL : 4;   // code words per lane
  constexpr int NFK = KT * KS, FK = (NFK + 3) / 4;                       // bf16 key (value) fragments, per warp
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) unsigned long long bar_stage[VF_STAGES], bar_stfree[VF_STAGES], bar_s, bar_sfree, bar_sk[2],
      bar_keys[2], bar_built[2], bar_p[2], bar_o[2];
  __shared__ unsigned s_tmem;
  __shared__ __align__(16) float s_vs[2][W];   // 2-bit window: 4 s_V per token
  __shared__ __align__(16) float s_vz[2][W];   // and z_V - 4 s_V
  __shared__ int s_abort;
  __shared__ int s_stage_cnt[VF_STAGES];   // copies issued into a stage

  const State& st = p.st;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.x, split = blockIdx.y;
  const long long gu = (long long)p.layer * st.units + u;
  const int G = st.G;
  const Geo g{D, W};
  const LayerView lv = layer_view(g, st.ldev[p.layer]);
  const int L = lv.L, nbw = lv.nbw, nq = lv.nq;
  const int b0 = (int)((long long)split * nbw / p.splits), b1 = (int)((long long)(split + 1) * nbw / p.splits);
  const int q0 = (int)((long long)split * nq / p.splits), q1 = (int)((long long)(split + 1) * nq / p.splits);
  const int nbc = b1 - b0, nqc = q1 - q0, nchunk = nbc + nqc;
  const unsigned sbase = smem_u32(smem);
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(S::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    // commit barriers take one arrival; the others one per warp of the producing group, after
    // the warp's own __syncwarp
    for (int i = 0; i < VF_STAGES; ++i) {
      mbar_init(smem_u32(&bar_stage[i]), 1);
      mbar_init(smem_u32(&bar_stfree[i]), 4);
      s_stage_cnt[i] = 0;
    }
    mbar_init(smem_u32(&bar_s), 1);
    mbar_init(smem_u32(&bar_sfree), 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bar_sk[i]), 1);
      mbar_init(smem_u32(&bar_keys[i]), 4);
      mbar_init(smem_u32(&bar_built[i]), 4);
      mbar_init(smem_u32(&bar_p[i]), 4);
      mbar_init(smem_u32(&bar_o[i]), 1);
    }
    mbar_fence_init();
    s_abort = 0;
  }
  // Q rows (zero beyond R), once
  {
    const int b = u / st.Hkv, kvh = u - b * st.Hkv, B = st.units / st.Hkv;
    for (int i = tid; i < VF_ROWS * (D / 2); i += VF_THREADS) {
      const int rr = i / (D / 2), c = 2 * (i - rr * (D / 2));
      unsigned val = 0u;
      if (rr < p.R) {
        const int jj = rr / G, hh = rr - jj * G;
        val = *reinterpret_cast<const unsigned*>(p.q + (((size_t)jj * B + b) * st.Hq + kvh * G + hh) * D + c);
      }
      *reinterpret_cast<unsigned*>(smem + vf_canon(rr, c, D)) = val;
    }
  }
  vf_proxy_fence();
  vf_fence_before();
  __syncthreads();
  vf_fence_after();
  const unsigned tS = s_tmem;                 // S: M = 64 rows, up to 3W columns
  const unsigned tO = s_tmem + S::TO_OFF;     // O: M = 64 rows, D columns

  // chunk c: bf16 entry b0 + c, then 2-bit entry q0 + (c - nbc)
  auto chunk_entry = [&](int c, int& eidx) -> int2 {
    if (c >= nchunk) {
      eidx = 0;
      return make_int2(0, -1);
    }
    if (c < nbc) {
      eidx = b0 + c;
      return st.blist[gu * st.capb + eidx];
    }
    const int qi = q0 + (c - nbc);
    eidx = nbw + qi;
    return st.qlist[gu * st.capq + qi];
  };

  if (warp == 8) {
    // ============================== tensor cores and copies (lane 0): S of chunk c, the refill of
    // the stage chunk c - 1 read, then P V of chunk c - 1
    if (lane == 0) {
      auto issue_copy = [&](int i, int2 e) {   // 2-bit chunk i of this split into stage i % VF_STAGES
        if (e.y < 0 || e.y >= st.capq) return;   // reported by the builders when they reach it
        const int sidx = i % VF_STAGES;
        const unsigned bar = smem_u32(&bar_stage[sidx]);
        s_stage_cnt[sidx] += 1;
        mbar_expect_tx(bar, S::QSLOT);
        bulk_g2s_hint(sbase + S::OFF_STG + sidx * S::STAGE, st.qslab + (gu * st.capq + e.y) * (long long)S::QSLOT,
                      S::QSLOT, bar, l2_evict_first_policy());
      };
      int ei;
      for (int i = 0; i < VF_STAGES && i < nqc; ++i) issue_copy(i, chunk_entry(nbc + i, ei));
      int2 refill = chunk_entry(nbc + VF_STAGES, ei);   // entry of the next refill, loaded ahead
      // descriptors of the operands' first K step; the next K step starts 256 bytes further, + 16
      // in the start-address field (16-byte units; shared addresses stay below 2^18 bytes); buffer
      // 1 lies a fixed distance after buffer 0
      const unsigned long long dQ = vf_desc(sbase, D * 16);
      const unsigned long long dK0 = vf_desc(sbase + S::OFF_BK, D * 16), dV0 = vf_desc(sbase + S::OFF_BV, W * 16),
                               dP0 = vf_desc(sbase + S::OFF_AP, S::KP * 16);
      int s_done = 0, pv_done = 0;   // launches issued
      for (int c = 0; c <= nchunk; ++c) {
        if (c < nchunk) {
          const int b = c & 1;
          bool ok = vf_wait(smem_u32(&bar_keys[b]), (c >> 1) & 1, st.err, abort_flag);
          if (ok && c >= 1) ok = vf_wait(smem_u32(&bar_sfree), (c - 1) & 1, st.err, abort_flag);
          if (!ok) break;
          vf_fence_after();
          const unsigned idesc = c >= nbc ? vf_idesc(VF_ROWS, 3 * W) : vf_idesc(VF_ROWS, W);
          const unsigned long long dK = dK0 + (unsigned)(b * (S::SBK >> 4));
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) vf_mma(tS, dQ + 16 * ks, dK + 16 * ks, idesc, ks > 0);
          vf_commit(smem_u32(&bar_s));       // for the softmax
          vf_commit(smem_u32(&bar_sk[b]));   // for the builders: key buffer b free again
          ++s_done;
        }
        // the builders finished the stage of chunk c - 1 before they wrote chunk c's keys: refill
        // it now, three 2-bit chunks ahead
        if (c >= 1) {
          const int qi = c - 1 - nbc;
          if (qi >= 0 && qi + VF_STAGES < nqc) {
            if (!vf_wait(smem_u32(&bar_stfree[qi % VF_STAGES]), (qi / VF_STAGES) & 1, st.err, abort_flag)) break;
            issue_copy(qi + VF_STAGES, refill);
            refill = chunk_entry(nbc + qi + VF_STAGES + 1, ei);
          }
        }
        if (c >= 1) {
          const int cc = c - 1, b = cc & 1;
          if (!vf_wait(smem_u32(&bar_p[b]), (cc >> 1) & 1, st.err, abort_flag)) break;
          vf_fence_after();
          // O += P V: M = 64 rows (A = P, both parts along K), N = D channels (B = values)
          constexpr unsigned idesc = vf_idesc(VF_ROWS, D);
          const unsigned long long dV = dV0 + (unsigned)(b * (S::SBV >> 4)), dP = dP0 + (unsigned)(b * (S::SAP >> 4));
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int kt = 0; kt < KT; ++kt)
              vf_mma(tO, dP + 16 * (part * KT + kt), dV + 16 * kt, idesc, cc > 0 || part > 0 || kt > 0);
          vf_commit(smem_u32(&bar_o[b]));
          ++pv_done;
        }
      }
      // the tensor-core work issued must finish before tensor memory is read or freed
      if (s_done > 0) vf_drain(smem_u32(&bar_s), (s_done - 1) & 1, st.err);
      if (pv_done > 0) vf_drain(smem_u32(&bar_o[(pv_done - 1) & 1]), ((pv_done - 1) >> 1) & 1, st.err);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============================== operand builders (warps 4-7), each on its own share of a chunk
    const int bw = warp - 4, tt = lane & 3;
    int eidx_n;
    int2 ent_n = chunk_entry(0, eidx_n);   // the next chunk's entry, loaded a chunk ahead
    // a bf16 slot's fragments (512 bytes each: one lane's 16 bytes, rows g, g + 8 at columns 2t,
    // 2t + 8; keys have tokens as rows, values channels), this warp's share, loaded ahead: the
    // keys of chunk c + 1 while chunk c's values are built, its values after those
    uint4 xk[FK], xv[FK];
    const unsigned long long ef = l2_evict_first_policy();   // the slots are read once per call
    auto load_bf16 = [&](int2 e, bool values, uint4 (&x)[FK]) {
      if (e.y < 0 || e.y >= st.capb) return;
      const uint8_t* slot = st.bslab + (gu * st.capb + e.y) * (long long)S::BSLOT + (values ? 32 * D : 0);
#pragma unroll
      for (int k = 0; k < FK; ++k) {
        const int ff = bw + 4 * k;
        if (ff < NFK) x[k] = ldg_hint(reinterpret_cast<const uint4*>(slot + (ff / KS) * (64 * D) + (ff % KS) * 512) + lane, ef);
      }
    };
    if (nbc > 0) {
      load_bf16(ent_n, false, xk);
      load_bf16(ent_n, true, xv);
    }
    for (int c = 0; c < nchunk; ++c) {
      const int b = c & 1;
      const int2 ent = ent_n;
      const bool is_q = c >= nbc;
      const int qi = c - nbc;
      ent_n = chunk_entry(c + 1, eidx_n);
      const bool slot_ok = ent.y >= 0 && ent.y < (is_q ? st.capq : st.capb);
      if (!slot_ok) {
        if (lane == 0) {
          atomicOr(st.err, ERR_TABLE);
          *abort_flag = 1;
        }
        break;
      }
      // keys of buffer b: their last reader, S of chunk c - 2, must be complete (every wait's
      // outcome is made uniform across the warp: its stores are collective)
      if (c >= 2 && !__all_sync(0xffffffffu, vf_wait(smem_u32(&bar_sk[b]), ((c - 2) >> 1) & 1, st.err, abort_flag)))
        break;
      if (is_q &&
          !__all_sync(0xffffffffu, vf_wait(smem_u32(&bar_stage[qi % VF_STAGES]), (qi / VF_STAGES) & 1, st.err, abort_flag)))
        break;
      const unsigned sBK = sbase + S::OFF_BK + b * S::SBK, sBV = sbase + S::OFF_BV + b * S::SBV;
      const uint8_t* sp = smem + S::OFF_STG + (qi % VF_STAGES) * S::STAGE;   // 2-bit chunk's stage
      auto word_at = [&](int byte0, int wj) -> unsigned {   // this lane's word wj of a code block
        return *reinterpret_cast<const unsigned*>(sp + byte0 + ((wj / CW) * 32 + lane) * (CW * 4) + (wj % CW) * 4);
      };
      auto store_bf16 = [&](bool values, const uint4 (&x)[FK]) {   // matrix k: rows + 8 (k & 1) + row, columns + 8 (k >> 1)
        const int m = lane >> 3;
#pragma unroll
        for (int k = 0; k < FK; ++k) {
          const int ff = bw + 4 * k;
          if (ff < NFK) {
            const int sub = ff / KS, blk = ff % KS;
            const unsigned dst = values
                                     ? sBV + vf_canon(16 * blk + 8 * (m & 1) + (lane & 7), 16 * sub + 8 * (m >> 1), W)
                                     : sBK + vf_canon(16 * sub + 8 * (m & 1) + (lane & 7), 16 * blk + 8 * (m >> 1), D);
            vf_stmatrix4(dst, x[k].x, x[k].y, x[k].z, x[k].w);
          }
        }
      };
      // ---- keys
      if (!is_q) {
        store_bf16(false, xk);
        if (c + 1 < nbc) load_bf16(ent_n, false, xk);
      } else if (bw < WPL) {
        // word wj holds fragments 2 wj, 2 wj + 1 (token tile mt, channel steps ks, ks + 1); a
        // warp's words share ks, so the warp needs the 32 channels 16 ks .. 16 ks + 31 only:
        // its own table of them, per channel and code the three bf16 parts of code * s + z (one
        // float32 fma, as the oracle dequantizes; truncated, truncated remainder, rest), laid out
        // [channel parity][16 channel pairs][4 codes] x 8 bytes so that a lookup instruction's
        // four lane groups (tt) read four disjoint sets of eight banks
        const int ks = (2 * bw) % KS;
        uint8_t* tab = smem + S::OFF_TAB + bw * 1024;
        {
          const float* kmin = reinterpret_cast<const float*>(sp + g.off_kmin());
          const float* kscale = reinterpret_cast<const float*>(sp + g.off_kscale());
          const int ch = 16 * ks + lane;
          const float sc = kscale[kparam_pos(ch)], mn = kmin[kparam_pos(ch)];
          uint2 e4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float val = fmaf((float)k, sc, mn);
            const unsigned hb = __float_as_uint(val) & 0xFFFF0000u;
            const float r = val - __uint_as_float(hb);
            const unsigned mb = __float_as_uint(r) & 0xFFFF0000u;
            e4[k] = make_uint2(__byte_perm(hb, mb, 0x7632), pack_bf16x2_rz(r - __uint_as_float(mb), 0.f));
          }
          uint4* tdst = reinterpret_cast<uint4*>(tab + (lane & 1) * 512 + (lane >> 1) * 32);
          tdst[0] = make_uint4(e4[0].x, e4[0].y, e4[1].x, e4[1].y);
          tdst[1] = make_uint4(e4[2].x, e4[2].y, e4[3].x, e4[3].y);
        }
        __syncwarp();
        const uint8_t* tlane = tab + tt * 32;   // channel 16 ks + 2 tt, code 0; odd channel + 512, + 8 per code
        for (int wj = bw; wj < WPL; wj += 4) {
          const unsigned w = word_at(0, wj);
          const int mt = (2 * wj) / KS;
#pragma unroll
          for (int f = 0; f < 2; ++f) {
            unsigned hp[4], mp[4], lp[4];
#pragma unroll
            for (int reg = 0; reg < 4; ++reg) {
              // reg: token 16 mt + gg + 8 (reg & 1), channels 16 (ks + f) + 2 tt + 8 (reg >> 1) + {0, 1}
              const int sh = 8 * f + 2 * reg;
              const uint8_t* te = tlane + (8 * f + 4 * (reg >> 1)) * 32;   // channel pair (16 f + 8 (reg >> 1)) / 2 further
              const uint2 e0 = *reinterpret_cast<const uint2*>(te + (((w >> sh) & 3u) << 3));
              const uint2 e1 = *reinterpret_cast<const uint2*>(te + 512 + (((w >> (sh + 16)) & 3u) << 3));
              hp[reg] = __byte_perm(e0.x, e1.x, 0x5410);
              mp[reg] = __byte_perm(e0.x, e1.x, 0x7632);
              lp[reg] = __byte_perm(e0.y, e1.y, 0x5410);
            }
            const int m = lane >> 3;
            const unsigned dst = sBK + vf_canon(16 * mt + 8 * (m & 1) + (lane & 7), 16 * (ks + f) + 8 * (m >> 1), D);
            vf_stmatrix4(dst, hp[0], hp[1], hp[2], hp[3]);
            vf_stmatrix4(dst + W * D * 2, mp[0], mp[1], mp[2], mp[3]);       // part 2: rows W ..
            vf_stmatrix4(dst + 2 * W * D * 2, lp[0], lp[1], lp[2], lp[3]);   // part 3: rows 2W ..
          }
        }
      }
      vf_proxy_fence();
      __syncwarp();
      if (lane == 0) vf_arrive(smem_u32(&bar_keys[b]));
      // values of buffer b: their last reader, P V of chunk c - 2, must be complete (so are its
      // softmax, the last reader of the value parameters and of P buffer b)
      if (c >= 2 && !__all_sync(0xffffffffu, vf_wait(smem_u32(&bar_o[b]), ((c - 2) >> 1) & 1, st.err, abort_flag)))
        break;
      // ---- values
      if (!is_q) {
        store_bf16(true, xv);
        if (c + 1 < nbc) load_bf16(ent_n, true, xv);
      } else {
        // word wj holds fragments 2 wj, 2 wj + 1 (channel tile mc, token steps kt, kt + 1; with
        // one token step the second fragment is the next channel tile), as 1 + code / 4
        for (int wj = bw; wj < WPL; wj += 4) {
          const unsigned w = word_at(g.off_vcode(), wj);
          const int F0 = 2 * wj, mc = F0 / KT, kt = F0 % KT;
#pragma unroll
          for (int f = 0; f < 2; ++f) {
            const int mcf = KT >= 2 ? mc : mc + f, ktf = KT >= 2 ? kt + f : kt;
            unsigned r[4];
#pragma unroll
            for (int reg = 0; reg < 4; ++reg) {
              const unsigned xw = w >> (8 * f + 2 * reg);
              r[reg] = 0x3F803F80u | ((xw & 3u) << 5) | (((xw >> 16) & 3u) << 21);
            }
            // matrix k = reg: channels 16 mcf + 8 (k & 1) + row, tokens 16 ktf + 8 (k >> 1)
            const int m = lane >> 3;
            vf_stmatrix4(sBV + vf_canon(16 * mcf + 8 * (m & 1) + (lane & 7), 16 * ktf + 8 * (m >> 1), W), r[0], r[1],
                         r[2], r[3]);
          }
        }
        if (bw == 0)
          for (int t = lane; t < W; t += 32) {
            const float vsc = reinterpret_cast<const float*>(sp + g.off_vscale())[vparam_pos(g, t)];
            const float vmn = reinterpret_cast<const float*>(sp + g.off_vmin())[vparam_pos(g, t)];
            s_vs[b][t] = 4.f * vsc;
            s_vz[b][t] = vmn - 4.f * vsc;
          }
      }
      vf_proxy_fence();
      __syncwarp();
      if (lane == 0) {
        vf_arrive(smem_u32(&bar_built[b]));
        if (is_q) vf_arrive(smem_u32(&bar_stfree[qi % VF_STAGES]));   // done with the stage
      }
    }
  } else {
    // ============================== softmax (warps 0-3), each warp on its own 16 rows
    const int q4 = lane & 3;
    const int ra = 16 * warp + (lane >> 2), rb = ra + 8;   // this lane's rows
    const bool va = ra < p.R, vb = rb < p.R;
    const int jda = ra / G, jdb = rb / G;
    const unsigned lane_off = (unsigned)(32 * warp) << 16;
    float mref_a = -INFINITY, mref_b = -INFINITY, lsum_a = 0.f, lsum_b = 0.f, zs_a = 0.f, zs_b = 0.f;
    int c = 0;
    bool ok = true;
    int eidx_n;
    int2 ent_n = chunk_entry(0, eidx_n);   // the next chunk's entry, loaded a chunk ahead
    for (; c < nchunk; ++c) {
      const int b = c & 1;
      const int2 ent = ent_n;
      const int eidx = eidx_n;
      ent_n = chunk_entry(c + 1, eidx_n);
      const bool is_q = c >= nbc;
      const int win = ent.x;
      // S of this chunk (every wait's outcome is made uniform across the warp: the loads are
      // collective)
      ok = __all_sync(0xffffffffu, vf_wait(smem_u32(&bar_s), c & 1, st.err, abort_flag));
      if (!ok) break;
      // ---- logits of this lane's two rows: x[4 j + e] row a, x[4 j + 2 + e] row b, token 8 j + 2 q4 + e
      float x[4 * NB];
      {
        vf_fence_after();
        const unsigned tSl = tS + lane_off;
        unsigned v0[4 * NB];
        vf_ld_rows<NB>(tSl, v0);
        if (is_q) {
          unsigned v1[4 * NB];
          vf_ld_rows<NB>(tSl + W, v1);
          vf_wait_ld(v0);
          vf_wait_ld(v1);
#pragma unroll
          for (int i = 0; i < 4 * NB; ++i) x[i] = __uint_as_float(v0[i]) + __uint_as_float(v1[i]);
          vf_ld_rows<NB>(tSl + 2 * W, v1);
          vf_wait_ld(v1);
#pragma unroll
          for (int i = 0; i < 4 * NB; ++i) x[i] = (x[i] + __uint_as_float(v1[i])) * p.scale_log2;
        } else {
          vf_wait_ld(v0);
#pragma unroll
          for (int i = 0; i < 4 * NB; ++i) x[i] = __uint_as_float(v0[i]) * p.scale_log2;
        }
        vf_fence_before();
        __syncwarp();
        if (lane == 0) vf_arrive(smem_u32(&bar_sfree));   // tensor memory may take S of chunk c + 1
      }
      // valid tokens of the window for a row: [tmin, tmax); draft j sees positions < L0 + j + 1
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
      const int tmax_a = va ? min(hi, p.L0 + jda + 1 - pos0) : 0;
      const int tmax_b = vb ? min(hi, p.L0 + jdb + 1 - pos0) : 0;
      if (lo > 0 || tmax_a < W || tmax_b < W) {
#pragma unroll
        for (int j = 0; j < NB; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = 8 * j + 2 * q4 + e;
            if (t < lo || t >= tmax_a) x[4 * j + e] = -INFINITY;
            if (t < lo || t >= tmax_b) x[4 * j + 2 + e] = -INFINITY;
          }
      }
      float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        ma = fmaxf(ma, fmaxf(x[4 * j], x[4 * j + 1]));
        mb = fmaxf(mb, fmaxf(x[4 * j + 2], x[4 * j + 3]));
      }
      ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      const bool raise_a = ma > mref_a + 8.f, raise_b = mb > mref_b + 8.f;   // false for -inf
      const float alpha_a = (raise_a && mref_a != -INFINITY) ? ex2(mref_a - ma) : 1.f;
      const float alpha_b = (raise_b && mref_b != -INFINITY) ? ex2(mref_b - mb) : 1.f;
      if (__any_sync(0xffffffffu, alpha_a != 1.f || alpha_b != 1.f)) {
        // rescale this warp's rows of O: the previous chunk's P V must be complete
        if (!__all_sync(0xffffffffu,
                        vf_wait(smem_u32(&bar_o[(c - 1) & 1]), ((c - 1) >> 1) & 1, st.err, abort_flag))) {
          ok = false;
          break;
        }
        vf_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          unsigned o[16];
          vf_ld_rows<4>(tO + lane_off + c0, o);
          vf_wait_ld(o);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            o[4 * j] = __float_as_uint(__uint_as_float(o[4 * j]) * alpha_a);
            o[4 * j + 1] = __float_as_uint(__uint_as_float(o[4 * j + 1]) * alpha_a);
            o[4 * j + 2] = __float_as_uint(__uint_as_float(o[4 * j + 2]) * alpha_b);
            o[4 * j + 3] = __float_as_uint(__uint_as_float(o[4 * j + 3]) * alpha_b);
          }
          vf_st_rows4(tO + lane_off + c0, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      if (raise_a) {
        lsum_a *= alpha_a;
        zs_a *= alpha_a;
        mref_a = ma;
      }
      if (raise_b) {
        lsum_b *= alpha_b;
        zs_b *= alpha_b;
        mref_b = mb;
      }
      const float mua = mref_a == -INFINITY ? 0.f : mref_a, mub = mref_b == -INFINITY ? 0.f : mref_b;
      // operands and value parameters of this chunk; P buffer b is free (its previous reader,
      // the P V of chunk c - 2, finished before the builders marked this chunk's operands built)
      if (!__all_sync(0xffffffffu, vf_wait(smem_u32(&bar_built[b]), (c >> 1) & 1, st.err, abort_flag))) {
        ok = false;
        break;
      }
      // ---- P (times 4 s_V for a 2-bit window) in two bf16 parts, into buffer b: rows ra, rb,
      // K index token t (part 1) and W + t (part 2)
      float mass_a = 0.f, mass_b = 0.f;
      unsigned ph[4 * NB / 2], pl[4 * NB / 2];   // [2 j + h]: block j, row half h (a, b)
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int t = 8 * j + 2 * q4;
        float pa0 = ex2(x[4 * j] - mua), pa1 = ex2(x[4 * j + 1] - mua);
        float pb0 = ex2(x[4 * j + 2] - mub), pb1 = ex2(x[4 * j + 3] - mub);
        mass_a += pa0 + pa1;
        mass_b += pb0 + pb1;
        if (is_q) {
          const float2 vs = *reinterpret_cast<const float2*>(&s_vs[b][t]);
          const float2 vz = *reinterpret_cast<const float2*>(&s_vz[b][t]);
          zs_a = fmaf(pa0, vz.x, fmaf(pa1, vz.y, zs_a));
          zs_b = fmaf(pb0, vz.x, fmaf(pb1, vz.y, zs_b));
          pa0 *= vs.x;
          pa1 *= vs.y;
          pb0 *= vs.x;
          pb1 *= vs.y;
        }
        vf_split2_pair(pa0, pa1, ph[2 * j], pl[2 * j]);
        vf_split2_pair(pb0, pb1, ph[2 * j + 1], pl[2 * j + 1]);
      }
      {
        const unsigned sAP = sbase + S::OFF_AP + b * S::SAP;
        const int m = lane >> 3;
#pragma unroll
        for (int j = 0; j < NB; j += 2) {
          // matrix k: rows 16 warp + 8 (k & 1) + row, K columns 8 (j + (k >> 1)) (+ W for part 2)
          const unsigned dst = sAP + vf_canon(16 * warp + 8 * (m & 1) + (lane & 7), 8 * (j + (m >> 1)), S::KP);
          vf_stmatrix4(dst, ph[2 * j], ph[2 * j + 1], ph[2 * j + 2], ph[2 * j + 3]);
          vf_stmatrix4(dst + (W / 8) * 128, pl[2 * j], pl[2 * j + 1], pl[2 * j + 2], pl[2 * j + 3]);
        }
      }
      // P (and the rescale of O) ready for the tensor-core issuer
      vf_proxy_fence();
      vf_fence_before();
      __syncwarp();
      if (lane == 0) vf_arrive(smem_u32(&bar_p[b]));
      mass_a += __shfl_xor_sync(0xffffffffu, mass_a, 1);
      mass_b += __shfl_xor_sync(0xffffffffu, mass_b, 1);
      mass_a += __shfl_xor_sync(0xffffffffu, mass_a, 2);
      mass_b += __shfl_xor_sync(0xffffffffu, mass_b, 2);
      lsum_a += mass_a;   // the row's four lanes hold the same sums
      lsum_b += mass_b;
      if (q4 == 0) {
        float* lrow = p.lse + ((long long)u * p.ent_cap + eidx) * VF_ROWS;
        if (va) lrow[ra] = mass_a > 0.f ? mua + lg2(mass_a) : -INFINITY;
        if (vb) lrow[rb] = mass_b > 0.f ? mub + lg2(mass_b) : -INFINITY;
      }
    }
    // c = chunks whose P went to the issuer (all of them on a normal exit)
    if (ok && c > 0)
      ok = __all_sync(0xffffffffu, vf_wait(smem_u32(&bar_o[(c - 1) & 1]), ((c - 1) >> 1) & 1, st.err, abort_flag));
    if (ok) {
      vf_fence_after();
      zs_a += __shfl_xor_sync(0xffffffffu, zs_a, 1);   // per-lane shares of the row's offset sum
      zs_b += __shfl_xor_sync(0xffffffffu, zs_b, 1);
      zs_a += __shfl_xor_sync(0xffffffffu, zs_a, 2);
      zs_b += __shfl_xor_sync(0xffffffffu, zs_b, 2);
      const size_t pbase = ((size_t)u * p.splits + split) * VF_ROWS;
      if (q4 == 0) {
        if (va) p.part_ml[pbase + ra] = make_float2(mref_a, lsum_a);
        if (vb) p.part_ml[pbase + rb] = make_float2(mref_b, lsum_b);
      }
      // O: this lane's rows ra, rb, columns 8 j + 2 q4, +1 of each 8-column block
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        unsigned o[16];
        if (c > 0) {
          vf_ld_rows<4>(tO + lane_off + c0, o);
          vf_wait_ld(o);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = c0 + 8 * j + 2 * q4;
          if (va)
            *reinterpret_cast<float2*>(p.part_o + (pbase + ra) * D + col) =
                make_float2(__uint_as_float(o[4 * j]) + zs_a, __uint_as_float(o[4 * j + 1]) + zs_a);
          if (vb)
            *reinterpret_cast<float2*>(p.part_o + (pbase + rb) * D + col) =
                make_float2(__uint_as_float(o[4 * j + 2]) + zs_b, __uint_as_float(o[4 * j + 3]) + zs_b);
        }
      }
    }
  }
  vf_fence_before();
  __syncthreads();
  // copies still in flight (after an expired wait) land before the CTA leaves
  if (tid == 0)
    for (int i = 0; i < VF_STAGES; ++i)
      if (s_stage_cnt[i] > 0) vf_drain(smem_u32(&bar_stage[i]), (s_stage_cnt[i] - 1) & 1, st.err);
  if (warp == 0) {
    vf_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(s_tmem), "r"(S::TMEM_COLS) : "memory");
  }
}

// ------------------------------------------------------------------------------ combine
// One CTA per (unit, draft j): merge the splits of draft j's G rows into its outputs, and turn
// every window's per-row log2-sum-exp into draft j's window mass (summed over its G heads),
// written to delta[j][unit][window] for qe_verify_commit.
constexpr int VF_COMBINE_THREADS = 128;
constexpr int VF_MAX_SPLITS = 16;

template <int D>
__global__ void __launch_bounds__(VF_COMBINE_THREADS) qe_verify_combine_kernel(const VerifyParams p, void* out,
                                                                              int out_fp32, float* delta,
                                                                              long long qstride) {
  const State& st = p.st;
  const int u = blockIdx.x, j = blockIdx.y, tid = threadIdx.x;
  const int G = st.G, r0 = j * G;
  const long long gu = (long long)p.layer * st.units + u;
  __shared__ float s_sc[VF_ROWS][VF_MAX_SPLITS];
  __shared__ float s_inv[VF_ROWS], s_lse[VF_ROWS];
  const Geo g{D, st.geo.W};
  const LayerView lv = layer_view(g, st.ldev[p.layer]);
  // row statistics of the draft's G rows
  if (tid < G) {
    const float2* ml = p.part_ml + (size_t)u * p.splits * VF_ROWS + r0 + tid;
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
  // outputs: head h, channels c .. c + 3
  const int b = u / st.Hkv, kvh = u - b * st.Hkv;
  for (int i = tid; i < G * (D / 4); i += VF_COMBINE_THREADS) {
    const int hh = i / (D / 4), c = 4 * (i - hh * (D / 4));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.splits; ++s) {   // a split without mass for the row wrote zeros
      const float sc = s_sc[hh][s];
      const float4 v = *reinterpret_cast<const float4*>(p.part_o + (((size_t)u * p.splits + s) * VF_ROWS + r0 + hh) * D + c);
      acc.x = fmaf(v.x, sc, acc.x);
      acc.y = fmaf(v.y, sc, acc.y);
      acc.z = fmaf(v.z, sc, acc.z);
      acc.w = fmaf(v.w, sc, acc.w);
    }
    const float inv = s_inv[hh];
    const size_t oi = (((size_t)j * st.units / st.Hkv + b) * st.Hq + kvh * G + hh) * D + c;
    if (out_fp32) {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + oi) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + oi) =
          make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
  }
  // window masses of draft j
  const int nent = lv.nbw + lv.nq;
  for (int e = tid; e < nent; e += VF_COMBINE_THREADS) {
    const int2 ent = e < lv.nbw ? st.blist[gu * st.capb + e] : st.qlist[gu * st.capq + (e - lv.nbw)];
    if (ent.x < 0 || ent.x >= st.maxw) continue;   // the sink is not scored
    const float* ls = p.lse + ((long long)u * p.ent_cap + e) * VF_ROWS + r0;
    float dS = 0.f;
    for (int hh = 0; hh < G; ++hh) dS += ex2(ls[hh] - s_lse[hh]);
    delta[j * qstride + (long long)u * st.maxw + ent.x] = dS;
  }
}

// ------------------------------------------------------------------------------ launchers
template <int D, int W>
static cudaError_t vf_launch_t(const VerifyParams& p, cudaStream_t s) {
  using S = VfShape<D, W>;
  qe_verify_attn_kernel<D, W><<<dim3(p.st.units, p.splits), VF_THREADS, S::SMEM_REQ, s>>>(p);
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

cudaError_t launch_verify_attn(const VerifyParams& p, cudaStream_t s) {
  const int D = p.st.geo.D, W = p.st.geo.W;
  if (p.splits < 1 || p.splits > VF_MAX_SPLITS || p.R < 1 || p.R > VF_ROWS) return cudaErrorInvalidValue;
  if (D == 128 && W == 16) return vf_launch_t<128, 16>(p, s);
  if (D == 128 && W == 32) return vf_launch_t<128, 32>(p, s);
  if (D == 128 && W == 64) return vf_launch_t<128, 64>(p, s);
  if (D == 64 && W == 16) return vf_launch_t<64, 16>(p, s);
  if (D == 64 && W == 32) return vf_launch_t<64, 32>(p, s);
  if (D == 64 && W == 64) return vf_launch_t<64, 64>(p, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_verify_combine(const VerifyParams& p, void* out, int out_fp32, float* delta, long long qstride,
                                  cudaStream_t s) {
  if (p.splits < 1 || p.splits > VF_MAX_SPLITS || p.R < 1 || p.R > VF_ROWS) return cudaErrorInvalidValue;
  if (p.st.geo.D == 128)
    qe_verify_combine_kernel<128><<<dim3(p.st.units, p.n_q), VF_COMBINE_THREADS, 0, s>>>(p, out, out_fp32, delta, qstride);
  else if (p.st.geo.D == 64)
    qe_verify_combine_kernel<64><<<dim3(p.st.units, p.n_q), VF_COMBINE_THREADS, 0, s>>>(p, out, out_fp32, delta, qstride);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

int verify_ctas_per_sm(int D, int W) {
  if (D == 128 && W == 16) return VfShape<128, 16>::CTAS_PER_SM;
  if (D == 128 && W == 32) return VfShape<128, 32>::CTAS_PER_SM;
  if (D == 128 && W == 64) return VfShape<128, 64>::CTAS_PER_SM;
  if (D == 64 && W == 16) return VfShape<64, 16>::CTAS_PER_SM;
  if (D == 64 && W == 32) return VfShape<64, 32>::CTAS_PER_SM;
  if (D == 64 && W == 64) return VfShape<64, 64>::CTAS_PER_SM;
  return 1;
}

int verify_max_rows() { return VF_ROWS; }
int verify_min_drafts() { return 5; }
int verify_max_splits() { return VF_MAX_SPLITS; }

}  // namespace qe
