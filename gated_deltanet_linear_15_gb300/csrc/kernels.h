// Host-visible launch descriptors of the chunk kernels (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace gdn {

constexpr unsigned kFlagL2Norm = 1u;
constexpr unsigned kFlagSpOff = 2u;
constexpr unsigned kFlagWindowOff = 4u;
constexpr unsigned kFlagDebugWaitTimeout = 0x80000000u;  // test hook, see gdn.h
constexpr unsigned kFlagDebugPeerTimeout = 0x40000000u;  // test hook, see gdn.h

// Single-launch sequence parallelism (bf16, d = 128): one launch of a recurrent kernel runs pass A, the
// start-state fix-up and pass B.  Each CTA takes a ticket (an atomic counter) when it starts and runs the
// ticket-th item of the work lists that the fix-up mode scan built on the device, in this order: the pass-A items
// that some fix-up needs, the pass-B items whose start needs no fix-up, the fix-up row blocks, the pass-B
// items whose start is fixed up.  An item waits (bounded) only for items of lower tickets, which belong to
// CTAs that started earlier: fix-up blocks for their (sequence, head)'s pass-A items, fixed-up pass-B items
// for their fix-up blocks.  One schedule per direction.
struct Sched {
  int *hdr;                               // [0] ticket counter, [1] pass-A items, [2] pass-B items without
                                          // fix-up, [3] (sequence, head) pairs with a fix-up, [4] fixed-up pass-B items
  int *listA, *listBn, *listF, *listBf;   // (segment * H + head) * 2 + role; segment * H + head; n * H + head; as listBn
  int *needA, *doneA, *doneF;             // per (sequence, head): pass-A items, pass-A items done, fix-up blocks done
};
constexpr int SCHED_HDR = 8;              // ints of each header
constexpr int FIX_ROWS = 8;               // state rows per fix-up block

struct FwdArgs {
  const void *q, *k, *v;
  const float *g, *beta, *S0;
  void *o;
  float *ST;
  Plan plan;
  const float *gsum;  // [CH_max, H] per-chunk sum of g
  int *status;
  float *Ebuf, *Mbuf, *Sstart;  // [S_max, H, D, D]
  void *states;                 // [CH_max, H, D, D] state at every chunk start (fp16 / fp32), or NULL
  int H, Lseg, Lfirst;  // segment lengths in chunks (seg_begin)
  float scale;
  unsigned flags;
  int pass;  // 0: segment end states / transitions, 1: outputs (+ saves if set), 2: states only
  // bf16 with d = 128, in place of the gate scan: the chunk-local half writes the per-chunk gate sums to
  // gsum_out (when set) and, with modes, its last CTA runs the fix-up mode scan over the S_max segments
  float *gsum_out;
  int modes, S_max;
  // bf16 with d = 128: the chunk context, see T64_*, T128_*, TQ_*.  t64 and tqkv are always set: the
  // chunk-local half writes them and the recurrent half reads them.  t128 and nrm are set when the
  // context is kept for the backward (then the chunk-local half also writes Ahat, N and the norms, and
  // pass 1 the W^T, Ut^T tiles); with o == NULL pass 1 writes no output and only states and context
  void *t64, *t128, *tqkv;
  float *nrm;
  Sched sched;  // single-launch sequence parallelism when sched_on (pass then names the pass-B kind, 1 or 2)
  int sched_on;
  // bf16 with d = 128, pass 1 / 2 over bal_pairs (sequence, head) pairs of equal length with bal_ns segments each
  // (bal_pairs = 0: one CTA per (segment, head), grid (S_max, H)): a 1-D grid whose first bal_big CTAs take the
  // later segments one each and whose other CTAs share the first segments
  int bal_pairs, bal_ns, bal_big;
  // bf16 with d = 128, pass 0 with passA_items = 2 S_max H > 0: a 1-D grid of at most one CTA per SM whose
  // CTAs take the (segment, head, role) items t (role t & 1, segment (t / 2) % S_max, head (t / 2) / S_max)
  // by ticket (status word 4), so that a pass with no work, or little, is one short wave
  int passA_items;
};

// Chunk context tiles of every (chunk, head), fp16 row-major, written by the forward:
//   t64  [CH_max, H, 5, 64, 64]:  X1 = Ahat diag(beta), X2 = lower(diag(gp) Ahat diag(beta rgp)), Ahat,
//                                 P = diag(gp) tril(Q K^T) diag(rgp), N = K K^T (normalised keys)
//   t128 [CH_max, H, 2, 128, 64]: W^T with its token columns scaled by gam (rows d_k), Ut^T (rows d_v)
//   tqkv [CH_max, H, 3, 64, 128]: the operand forms of K, Q, V (normalised, q scaled, fp16; rows = tokens,
//                                 zero past the sequence end)
//   nrm  [CH_max, H, 2, 64] fp32: reciprocal norms 1/|k|, 1/|q| per token (1 without normalisation)
constexpr int T64_X1 = 0, T64_X2 = 1, T64_AH = 2, T64_P = 3, T64_N = 4, T64_TILES = 5;
constexpr int T128_W = 0, T128_U = 1, T128_TILES = 2;
constexpr int TQ_K = 0, TQ_Q = 1, TQ_V = 2, TQ_TILES = 3;
// Tiles the reverse chain leaves for the local-gradient kernel, fp16 row-major:
//   tc   [CH_max, H, 2, 128, 64]: dUt^T (rows d_v, columns token) and dO in its operand form (rows 0-63: tokens x
//                                 features 0-63, rows 64-127: tokens x features 64-127; zero past the sequence end)
constexpr int TC_DUT = 0, TC_DO = 1, TC_TILES = 2;

struct BwdArgs {
  const void *q, *k, *v, *dO;
  const float *g, *beta, *dST;
  void *dq, *dk, *dv;
  float *dg, *dbeta, *dS0;
  Plan plan;
  const float *gsum;
  int *status;
  float *Fbuf, *Rbuf, *dSend;  // [S_max, H, D, D]
  const void *states;          // [CH_max, H, D, D] forward state at each chunk start
  void *dstates;               // [CH_max, H, D, D] dS at each chunk end
  int H, Lseg, Lfirst;
  float scale;
  unsigned flags;
  int pass;  // reverse chain: 0 segment starts / transitions, 1 per-chunk dS
  const float *nrm;  // context reciprocal norms (bf16, d = 128), see FwdArgs
  Sched sched;       // single-launch sequence parallelism when sched_on, see FwdArgs
  int sched_on;
  int bal_pairs, bal_ns, bal_big;  // balanced chain over equal-length sequences, see FwdArgs
  int passA_items;                 // pass A by ticket (status word 5), see FwdArgs
  // local gradients over ord_n equal-length sequences of ord_nc chunks each: the chunks in the order of
  // their offset within the segment (lifo_chunk in bwd_local_tc.cu); 0: in chunk order
  int ord_n, ord_nc;
};

struct FixupArgs {
  Plan plan;
  const float *gsum;
  const float *E, *M;  // end states / transitions per (segment, head)
  float *out;          // corrected start (forward) or end (reverse) states
  int H, D, Lseg, Lfirst;
  unsigned flags;
  int reverse;
  const int *fixflag;  // nonzero iff some segment of this direction needs the fix-up (NULL: always run)
  int *status;         // status word (an expired wait for a step's inputs sets value 4), or NULL
  // NULL: grid (D / FIX_ROWS, H, N), one row block per CTA; else a 1-D grid whose CTAs take the row blocks
  // t (rb = t % (D / FIX_ROWS), then head, then sequence) by ticket from this zeroed counter
  int *ticket;
};

struct RecArgs {
  const void *q, *k, *v;  // [N, T, H, D] element type of the call
  const float *g, *beta;  // [N, T, H]
  const float *S_in;      // [N, H, D, D] or NULL (zeros)
  void *o;                // [N, T, H, D]
  float *S_out;           // [N, H, D, D], may equal S_in
  int T, H;
  float scale;
  unsigned flags;
};

// zero: `nzero` ints cleared with the status words (the schedules' counters), or NULL.  With gsum and modes
// set (the saved-context backward, which takes the forward's gate sums) the plan kernel also runs the fix-up
// mode scan and builds the schedules in sched[0] / sched[1] (hdr NULL: none) instead of the gate scan.
int launch_plan(const Plan &p, const int *cu, int N, int T, int Lseg, int Lfirst, int S_max, int CH_max, int *status,
                int *zero, int nzero, cudaStream_t st, const float *gsum = nullptr, int H = 0, int modes = 0,
                unsigned flags = 0, const Sched *sched = nullptr);
// sched[0] / sched[1]: forward / reverse schedules to build (hdr NULL: none)
int launch_gate_scan(const Plan &p, const float *g, int H, int CH_max, float *gsum, int *status, int modes, int Lseg,
                     int Lfirst, int S_max, unsigned flags, const Sched *sched, int NH, cudaStream_t st);
// ctas > 0 (with a.ticket set): that many CTAs take the row blocks by ticket
int launch_fixup(const FixupArgs &a, int N, int ctas, cudaStream_t st);

int launch_fwd_chunk(const FwdArgs &a, bool is_bf16, int D, dim3 grid, cudaStream_t st);
// tcgen05 forward for bf16 inputs and d = 128, chunk-local half: one CTA per (chunk, head) over CH_max x H;
// maps: q, k, v over [tokens, H, 128] bf16 (box 64 x 1 x 64), the t64 tiles ([rows, 64] fp16, box 64 x 64)
// and the tqkv tiles ([rows, 128] fp16, box 64 x 64)
int launch_fwd_prep_tc(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &t64, const CUtensorMap &tqkv, int CH_max, cudaStream_t st);
// tcgen05 forward, recurrent half: one CTA per (segment, head); reads the tqkv and t64 tiles, stores the
// chunk-start states ([rows, 128] fp16, box 64 x 128), the t128 tiles ([rows, 64] fp16, box 64 x 128) and
// full chunks of o (map over [tokens, H, 128] bf16, box 64 x 1 x 64)
int launch_fwd_tc(const FwdArgs &a, const CUtensorMap &tqkv, const CUtensorMap &t64, const CUtensorMap &ts,
                  const CUtensorMap &t128, const CUtensorMap &to, dim3 grid, cudaStream_t st);
int launch_bwd_chain(const BwdArgs &a, bool is_bf16, int D, dim3 grid, cudaStream_t st);
// tcgen05 reverse chain (bf16, d = 128); maps: the tqkv context ([rows, 128] fp16, box 64x64), dO
// ([tokens, H, 128] bf16, box 64x1x64), the t64 and t128 context tiles, and the per-chunk dS store
// ([rows, 128] fp16, box 64x128x1)
int launch_bwd_chain_tc(const BwdArgs &a, const CUtensorMap *maps, dim3 grid, cudaStream_t st);
int launch_bwd_local(const BwdArgs &a, bool is_bf16, int D, int CH_max, cudaStream_t st);
// tcgen05 local-gradient kernel (bf16, d = 128); maps: the tqkv context, dO ([tokens, H, 128] bf16, box
// 64x1x64), the fp16 per-chunk states S0 and dS ([rows, 128] as a 3-D map, box 64x128x1), the t64 and t128
// context tiles, and dq, dk, dv (as dO)
int launch_bwd_local_tc(const BwdArgs &a, const CUtensorMap *maps, int CH_max, cudaStream_t st);
// token-by-token forward over NH = N * H (sequence, head) pairs
int launch_recurrent(const RecArgs &a, bool is_bf16, int D, int NH, cudaStream_t st);

}  // namespace gdn
