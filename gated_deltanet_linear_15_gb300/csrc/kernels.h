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
  int H, Lseg;
  float scale;
  unsigned flags;
  int pass;  // 0: segment end states / transitions, 1: outputs (+ states if set), 2: states only
  const void *wy;  // precomputed WY tiles (backward only) or NULL: X1/X2 come by TMA, no inverse
  void *wy_save;   // outputs pass (bf16, d = 128): also write the inline X1, X2, Ahat tiles here, or NULL
};

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
  int H, Lseg;
  float scale;
  unsigned flags;
  int pass;  // reverse chain: 0 segment starts / transitions, 1 per-chunk dS
  const void *wy;  // precomputed WY tiles or NULL
};

struct FixupArgs {
  Plan plan;
  const float *gsum;
  const float *E, *M;  // end states / transitions per (segment, head)
  float *out;          // corrected start (forward) or end (reverse) states
  int H, D, Lseg;
  unsigned flags;
  int reverse;
  const int *fixflag;  // nonzero iff some segment of this direction needs the fix-up (NULL: always run)
};

// WY tiles of every (chunk, head): fp16 [CH_max, H, 3, 64, 64] = X1, X2, Ahat (row-major)
struct WyArgs {
  const void *k;
  const float *g, *beta;
  Plan plan;
  void *wy;
  int *status;
  int H;
  unsigned flags;
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

int launch_plan(const Plan &p, const int *cu, int N, int T, int Lseg, int S_max, int CH_max, int *status,
                cudaStream_t st);
int launch_gate_scan(const Plan &p, const float *g, int H, int CH_max, float *gsum, int *status, int modes, int Lseg,
                     int S_max, unsigned flags, cudaStream_t st);
int launch_fixup(const FixupArgs &a, int N, cudaStream_t st);

int launch_fwd_chunk(const FwdArgs &a, bool is_bf16, int D, dim3 grid, cudaStream_t st);
// tcgen05 forward for bf16 inputs and d = 128; q, k, v tensor maps over [tokens, H, 128] with a 64 x 1 x 64 box;
// tw: the WY tiles as [rows, 64] fp16 with a 64 x 64 box (used when a.wy != NULL)
int launch_fwd_tc(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                  const CUtensorMap &tw, const CUtensorMap &ts, dim3 grid, cudaStream_t st);
int launch_wy(const WyArgs &a, int CH_max, cudaStream_t st);
int launch_bwd_chain(const BwdArgs &a, bool is_bf16, int D, dim3 grid, cudaStream_t st);
// tcgen05 reverse chain (bf16, d = 128); maps: q, k, dO ([tokens, H, 128] bf16, box 64x1x64) and the WY tiles
int launch_bwd_chain_tc(const BwdArgs &a, const CUtensorMap *maps, dim3 grid, cudaStream_t st);
int launch_bwd_local(const BwdArgs &a, bool is_bf16, int D, int CH_max, cudaStream_t st);
// tcgen05 local-gradient kernel (bf16, d = 128); maps: q, k, v, dO ([tokens, H, 128] bf16, box 64x1x64) and
// the fp16 per-chunk states S0 and dS ([rows, 128] as a 3-D map, box 64x128x1), and the WY tiles
int launch_bwd_local_tc(const BwdArgs &a, const CUtensorMap *maps, int CH_max, cudaStream_t st);
// token-by-token forward over NH = N * H (sequence, head) pairs
int launch_recurrent(const RecArgs &a, bool is_bf16, int D, int NH, cudaStream_t st);

}  // namespace gdn
