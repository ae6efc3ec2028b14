// qe_tok.cuh -- the five-tier per-token cache (HqeKV reading notes, §3.1: every cached pair is
// kept in BF16, 4-bit or 2-bit uniform (eq. (2)), 1-bit normal (eqs. (3)-(4)), or evicted).
//
// Layout on the device (per layer, per unit u = (batch element, KV head)):
//  * four ranked pools, one per kept tier, each a run of 16-token tiles ordered by position;
//  * a tail of BF16 tiles holding the sink, the recent tokens and every token appended since the
//    last re-rank (ordered by position);
//  * each pool and the tail exist twice (buffers 0 and 1): a re-rank reads one and writes the
//    other, then the layer switches;
//  * per token of every pool: its position (int32) and its score (float32).
// Tiles are stored in mma fragment order so the attention streams them with one bulk copy and
// unpacks codes in registers:
//  * BF16 tile (64 D bytes): K then V, the layout of the window path's 16-token sub-tile;
//  * b-bit tile (4 D b + 256 bytes): key codes, value codes (2 D b bytes each), then the key
//    parameters and the value parameters, one float2 per token: (min, scale) for the uniform
//    tiers, (mean, std) for the normal one.
//    Code layout: lane l of the m16n8k16 A fragment holds, per 16-channel step (keys) or
//    16-channel block (values, A = V^T), eight codes in its four registers r (two halves each);
//    a 32-bit word carries 4 / b steps: the low-half code of step k (inside the word) and
//    register r at bit b (4 k + r), the high-half code 16 bits above.  One shift and one and-or
//    then yield a register's two operands 1 + code / 2^b.
#pragma once

#include <cstdint>

#include "qe_common.cuh"

namespace qe {

enum : int { TK_BF16 = 0, TK_INT4 = 1, TK_INT2 = 2, TK_NQ1 = 3, TK_EVICT = 4, TK_TAIL = 5 };

QE_HD int tk_bits(int z) { return z == TK_INT4 ? 4 : z == TK_INT2 ? 2 : 1; }

struct TokGeo {
  int D;
  QE_HD int bf_tile() const { return 64 * D; }
  QE_HD int code_bytes(int b) const { return 2 * D * b; }            // one block (K or V), 16 tokens
  QE_HD int q_tile(int b) const { return 4 * D * b + 256; }
  QE_HD int off_vcode(int b) const { return 2 * D * b; }
  QE_HD int off_kpar(int b) const { return 4 * D * b; }
  QE_HD int off_vpar(int b) const { return 4 * D * b + 128; }
  QE_HD int wpl(int b) const { return D * b / 64; }                  // code words per lane per block
  QE_HD int cw(int b) const { return wpl(b) < 4 ? wpl(b) : 4; }      // words per lane per chunk
};

// Byte offset (in its block) of the word holding a code, and its bit position.
// step: key channel step (c / 16) or value channel block; row16 / col16: position inside the
// 16 x 16 A fragment (keys: row = token, column = channel; values: row = channel, column = token).
QE_HD CodePos tk_code_pos(const TokGeo& g, int b, int step, int row16, int col16) {
  const int lane = (row16 & 7) * 4 + ((col16 & 7) >> 1);
  const int reg = (row16 >> 3) + 2 * (col16 >> 3);
  const int half = col16 & 1;
  const int per_word = 4 / b;
  const int j = step / per_word, k = step - j * per_word;
  const int cw = g.cw(b);
  CodePos p;
  p.byte = ((j / cw) * 32 + lane) * (cw * 4) + (j % cw) * 4;
  p.bit = 16 * half + b * (4 * k + reg);
  return p;
}
QE_HD CodePos tk_kcode_pos(const TokGeo& g, int b, int tok, int c) { return tk_code_pos(g, b, c >> 4, tok, c & 15); }
QE_HD CodePos tk_vcode_pos(const TokGeo& g, int b, int tok, int c) {
  CodePos p = tk_code_pos(g, b, c >> 4, c & 15, tok);
  p.byte += g.off_vcode(b);
  return p;
}

// Per-layer dynamic header (device resident, updated by the kernels).
struct TokLayer {
  int L;          // tokens appended
  int n_tail;     // tokens in the tail (uniform over units)
  int buf;        // current buffer of the pools and the tail
  int step;       // decode steps since the last re-rank
  int pend;       // appended tokens whose length is committed by the next combine
  int pad[3];
};

struct TokState {
  TokGeo g;
  int units, G, Hkv, Hq;
  int n_sink, n_recent, max_context, period, score_window;
  int cap[4];              // ranked pool capacities (tokens, multiples of 16) per kept tier
  int cap_tail;            // tail capacity (tokens, multiple of 16)
  int cost[5];             // attention cost of one tile: BF16, INT4, INT2, 1-bit, tail (BF16)
  double frac[4];          // token fractions of BF16 (sink and recent included), INT4, INT2, 1-bit
  // pools: [layer][buf][unit][cap tiles] tiles; positions and scores [layer][buf][unit][cap]
  uint8_t* pool[4];
  int* pos[4];
  float* score[4];
  uint8_t* tail;
  int* tail_pos;
  float* tail_score;
  TokLayer* hdr;           // [layers]
  int* cnt;                // [layers][units][4] ranked pool counts
  long long* cum;          // [layers][units + 1] ranked cost prefix
  unsigned* err;
  // re-rank scratch, [layers][units][max_context] each: one slot per layer of a call, which
  // re-ranks a run of layers in one launch (slot = layer - first layer of the run)
  unsigned long long* ckey;
  int* csrc;
  uint8_t* newt;
  int* order;              // [layers][units][4][max_context]
  int* src_of;             // [layers][units][max_context]
  int* ncnt;               // [layers][units][4] ranked pool counts after the re-rank being applied
  unsigned* done;          // [layers] combine completion counters
};

QE_HD long long tk_pool_tile_index(const TokState& s, int z, int layer, int buf, int u) {
  return (((long long)layer * 2 + buf) * s.units + u) * (s.cap[z] / 16);
}
QE_HD long long tk_pool_tok_index(const TokState& s, int z, int layer, int buf, int u) {
  return (((long long)layer * 2 + buf) * s.units + u) * s.cap[z];
}
QE_HD long long tk_tail_tok_index(const TokState& s, int layer, int buf, int u) {
  return (((long long)layer * 2 + buf) * s.units + u) * s.cap_tail;
}
QE_HD int tk_tile_bytes(const TokState& s, int z) {
  return z == TK_BF16 || z == TK_TAIL ? s.g.bf_tile() : s.g.q_tile(tk_bits(z));
}

// One round of the warp's 32-way search for the largest u in [lo, hi] with X(u) <= x (X
// nondecreasing, X(lo) <= x): lane l tests unit search32_unit(lo, hi, l); with m the last lane
// whose unit passed, the answer lies in [unit(m), unit(m + 1) - 1], or [unit(31), hi] for
// m = 31 (search32_narrow).  Each round shrinks the interval about 32-fold.
QE_HD int search32_unit(int lo, int hi, int lane) { return lo + (int)(((long long)lane * (hi - lo + 1)) >> 5); }
QE_HD void search32_narrow(int& lo, int& hi, int m) {
  const int s = hi - lo + 1;
  const int n_lo = lo + (int)(((long long)m * s) >> 5);
  hi = m == 31 ? hi : lo + (int)(((long long)(m + 1) * s) >> 5) - 1;
  lo = n_lo;
}

}  // namespace qe
