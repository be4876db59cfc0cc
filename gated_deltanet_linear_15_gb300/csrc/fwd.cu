// Fused chunked forward of the gated delta rule over one segment of one
// (sequence, head): WY stage, chunk-to-chunk state pass and output in one
// kernel, so W, U, the corrected values and the per-chunk state never reach
// HBM (onedev.kr FlashQLA talk summary, paragraph on the WY representation:
// four steps, of which FLA writes W, U, S to HBM between operators).
//
// Per chunk (C = 64 tokens, S is d_v x d_k, G = in-chunk prefix of g):
//   N    = strict_tril(K K^T);  Ahat = (I + diag(beta) N)^{-1}      (fp32)
//   W    = diag(gam) Ahat diag(beta) K;   U = (diag(gp) Ahat diag(beta rgp)) V
//   Ut   = U - W S0^T                                    (corrected values)
//   O    = diag(gam) Q S0^T + P Ut,  P = diag(gp) tril_incl(Q K^T) diag(rgp)
//   S_C  = gam_C S0 + Ut^T diag(cdec) K
// The state lives in fp32 registers for the whole segment; its bf16 copy in
// shared memory is the MMA operand of the next chunk.
//
// Passes (one CTA per (segment, head[, role])):
//   pass A: segments whose successor needs a corrected start: run from the
//           segment's own start (initial state, warm-up, or zero) and store the
//           end state E; role 1 runs the same recurrence with v = 0 from I to
//           give the d_k x d_k transition M (onedev.kr talk summary, paragraph
//           on parallelism: zero-state recursion plus one d_k x d_k correction).
//   pass B: every segment from its exact start, writing O (and S_T).
//   pass S: as pass B but writing the bf16 state at every chunk start instead
//           of O (input of the backward).
#include "chunk_common.cuh"
#include "kernels.h"

namespace gdn {

template <typename E, int D> struct FwdSmem {
  static constexpr int LD = D + Pad<E>::v;
  static constexpr int LC = CH + Pad<E>::v;
  static constexpr int LN = CH + 4;
  E q[CH * LD], k[CH * LD], v[CH * LD], kt[CH * LD], w[CH * LD], ut[CH * LD];
  E s[D * LD];
  E p[CH * LC], x1[CH * LC], x2[CH * LC];
  float nf[CH * LN];
  float g[CH], beta[CH];
  Gates gt;
  float ys[1152];
};

template <typename I, int D>
__global__ void __launch_bounds__(NTHREADS, 1) fwd_chunk_kernel(FwdArgs a) {
  using E = typename OpType<I>::T;
  using SM = FwdSmem<E, D>;
  constexpr int LD = SM::LD, LC = SM::LC, LN = SM::LN;
  constexpr int SWM = D / 4, SWN = D / 2;  // state / output warp tile
  extern __shared__ __align__(128) unsigned char smraw[];
  SM &sm = *reinterpret_cast<SM *>(smraw);

  const int s = blockIdx.x, h = blockIdx.y, role = blockIdx.z;
  // pass A of a call in which no segment needs the exact fix-up (status[1], set by the fix-up mode scan)
  if (a.pass == 0 && a.status && a.status[1] == 0) return;
  const int H = a.H;
  const int n = a.plan.seg_seq[s];
  if (n < 0) return;
  const int j = s - a.plan.seq_seg0[n], nseg = a.plan.seq_nseg[n];
  const int len = a.plan.seq_len[n], chunk0 = a.plan.seq_chunk0[n];
  const long bos = a.plan.seq_bos[n];
  const int nchunks = (len + CH - 1) / CH;
  const int cbeg = seg_begin(j, a.Lfirst, a.Lseg), cend = min(seg_begin(j + 1, a.Lfirst, a.Lseg), nchunks);
  const bool window = !(a.flags & kFlagWindowOff);
  int w = 0;
  const int mode = fwd_start_mode(a.gsum, H, h, chunk0, cbeg, j, window, &w);
  bool transition = false;
  if (a.pass == 0) {
    if (j >= nseg - 1) return;
    int w2;
    if (fwd_start_mode(a.gsum, H, h, chunk0, cend, j + 1, window, &w2) != START_FIXUP) return;
    if (role == 1) {
      if (mode != START_FIXUP) return;
      transition = true;
    }
  } else if (role != 0) {
    return;
  }
  const bool outputs = (a.pass == 1);
  const bool need_v = !transition;
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = warp >> 1, wc = warp & 1;

  const I *qg = static_cast<const I *>(a.q);
  const I *kg = static_cast<const I *>(a.k);
  const I *vg = static_cast<const I *>(a.v);
  const size_t DD = (size_t)D * D;
  const size_t sh_idx = (size_t)s * H + h;

  int cfirst = cbeg;
  if (mode == START_WARMUP && !transition) cfirst = cbeg - w;

  auto issue_loads = [&](int c) {
    const long tok0 = bos + (long)c * CH;
    const int nvalid = min(CH, len - c * CH);
    load_tile<I, D>(sm.k, LD, kg, H, h, tok0, nvalid);
    if (need_v) load_tile<I, D>(sm.v, LD, vg, H, h, tok0, nvalid);
    if (outputs && c >= cbeg) load_tile<I, D>(sm.q, LD, qg, H, h, tok0, nvalid);
    load_scalars(sm.g, a.g, H, h, tok0, nvalid, 0);
    load_scalars(sm.beta, a.beta, H, h, tok0, nvalid, 64);
    cp_async_commit();
  };

  issue_loads(cfirst);

  // ---- initial state into registers (fp32) and its E copy
  Acc<SWM, SWN> Sacc;
  bool nbad = false;  // numeric guard: an fp16 operand out of range
  {
    const float *src = nullptr;
    if (transition) {
      src = nullptr;
    } else if (mode == START_INIT) {
      src = a.S0 ? a.S0 + ((size_t)n * H + h) * DD : nullptr;
    } else if (mode == START_FIXUP && a.pass != 0) {
      src = a.Sstart + sh_idx * DD;
    }
    const int m0 = wr * SWM, n0 = wc * SWN;
    Sacc.pairs([&](int r, int c, float &v0, float &v1) {
      const int row = m0 + r, col = n0 + c;
      if (src) {
        const float2 t = *reinterpret_cast<const float2 *>(src + (size_t)row * D + col);
        v0 = t.x;
        v1 = t.y;
      } else if (transition) {
        v0 = (row == col) ? 1.f : 0.f;
        v1 = (row == col + 1) ? 1.f : 0.f;
      } else {
        v0 = v1 = 0.f;
      }
      st2(&sm.s[row * LD + col], v0, v1);
    });
  }

  Acc<32, SWN> X;  // U / Ut (warps 0-3) or the output (warps 4-7)

  for (int c = cfirst; c < cend; ++c) {
    const bool emit = outputs && c >= cbeg;
    const long tok0 = bos + (long)c * CH;
    const int nvalid = min(CH, len - c * CH);
    cp_async_wait_all();
    __syncthreads();  // tiles of chunk c landed; state copy of S0 complete

    if (a.pass != 0 && a.states && c >= cbeg) {
      // bf16/fp32 copy of the state at the chunk start, for the backward
      E *dst = static_cast<E *>(a.states) + ((size_t)(chunk0 + c) * H + h) * DD;
      constexpr int EPV = 16 / sizeof(E);
      for (int e = threadIdx.x; e < D * D / EPV; e += NTHREADS) {
        const int r = e / (D / EPV), cc = (e % (D / EPV)) * EPV;
        *reinterpret_cast<uint4 *>(dst + (size_t)r * D + cc) = *reinterpret_cast<const uint4 *>(&sm.s[r * LD + cc]);
      }
    }
    nbad |= prep_rows<I, E, D>(sm.k, LD, 1.f, l2, nullptr);
    if (emit) nbad |= prep_rows<I, E, D>(sm.q, LD, a.scale, l2, nullptr);
    if (need_v) nbad |= prep_rows<I, E, D>(sm.v, LD, 1.f, false, nullptr);
    if (warp == 0) gate_prefix(sm.g, sm.gt);
    __syncthreads();

    // ---- K~ = diag(cdec) K, and [K; Q] K^T  ->  N (fp32) and P (E)
    for (int e = threadIdx.x; e < CH * D; e += NTHREADS) {
      const int r = e / D, cc = e % D;
      sm.kt[r * LD + cc] = fromf<E>(tof(sm.k[r * LD + cc]) * sm.gt.cdec[r]);
    }
    if (warp < 4 || emit) {
      Acc<32, 32> acc;
      acc.zero();
      const E *A = (warp < 4) ? sm.k : sm.q;
      const int m0 = (wr & 1) * 32, n0 = wc * 32;
      warp_mma<32, 32, false, false>(acc, A, LD, sm.k, LD, m0, n0, D);
      if (warp < 4) {
        acc.each([&](int r, int cc, float &v) {
          const int row = m0 + r, col = n0 + cc;
          if (col < row) sm.nf[row * LN + col] = v;
        });
      } else {
        acc.each([&](int r, int cc, float &v) {
          const int row = m0 + r, col = n0 + cc;
          sm.p[row * LC + col] = fromf<E>(col <= row ? v * gratio(sm.gt, row, col) : 0.f);
        });
      }
    }
    __syncthreads();

    wy_inverse<std::is_same<E, float>::value, false>(sm.nf, LN, sm.beta, sm.ys,
                                                     [&](int r, int c, float a0, float a1) {
      const float b0 = sm.beta[c], b1 = sm.beta[c + 1];
      st2(&sm.x1[r * LC + c], a0 * b0, a1 * b1);
      st2(&sm.x2[r * LC + c], c <= r ? a0 * b0 * gratio(sm.gt, r, c) : 0.f,
          c + 1 <= r ? a1 * b1 * gratio(sm.gt, r, c + 1) : 0.f);
    });

    // ---- U (warps 0-3, registers) and -W (warps 4-7, shared)
    {
      const int ww = warp & 3;
      const int m0 = (ww >> 1) * 32, n0 = (ww & 1) * SWN;
      if (warp < 4) {
        X.zero();
        if (need_v) warp_mma<32, SWN, false, true>(X, sm.x2, LC, sm.v, LD, m0, n0, CH);
      } else {
        Acc<32, SWN> acc;
        acc.zero();
        warp_mma<32, SWN, false, true>(acc, sm.x1, LC, sm.k, LD, m0, n0, CH);
        acc.pairs([&](int r, int cc, float &v0, float &v1) {
          const float gm = -sm.gt.gam[m0 + r];
          st2(&sm.w[(m0 + r) * LD + n0 + cc], v0 * gm, v1 * gm);
        });
      }
    }
    __syncthreads();

    // ---- Ut = U + (-W) S0^T (warps 0-3);  O1 = Q S0^T (warps 4-7)
    {
      const int ww = warp & 3;
      const int m0 = (ww >> 1) * 32, n0 = (ww & 1) * SWN;
      if (warp < 4) {
        warp_mma<32, SWN, false, false>(X, sm.w, LD, sm.s, LD, m0, n0, D);
      } else if (emit) {
        X.zero();
        warp_mma<32, SWN, false, false>(X, sm.q, LD, sm.s, LD, m0, n0, D);
      }
    }
    __syncthreads();

    if (c + 1 < cend) issue_loads(c + 1);  // Q, K, V, g, beta are free now

    if (warp < 4) {
      const int m0 = (warp >> 1) * 32, n0 = (warp & 1) * SWN;
      X.pairs([&](int r, int cc, float &v0, float &v1) { st2(&sm.ut[(m0 + r) * LD + n0 + cc], v0, v1); });
    }
    __syncthreads();

    // ---- S_C = gam_C S0 + Ut^T K~ (all warps);  O = diag(gam) O1 + P Ut (warps 4-7)
    {
      const float gC = sm.gt.gamC;
      Sacc.each([&](int r, int cc, float &v) { v *= gC; });
      warp_mma<SWM, SWN, true, true>(Sacc, sm.ut, LD, sm.kt, LD, wr * SWM, wc * SWN, CH);
      if (warp >= 4 && emit) {
        const int ww = warp & 3;
        const int m0 = (ww >> 1) * 32, n0 = (ww & 1) * SWN;
        X.each([&](int r, int cc, float &v) { v *= sm.gt.gam[m0 + r]; });
        warp_mma<32, SWN, false, true>(X, sm.p, LC, sm.ut, LD, m0, n0, CH);
        I *ostage = reinterpret_cast<I *>(sm.w);  // output staging in the input dtype
        X.pairs([&](int r, int cc, float &v0, float &v1) { st2(&ostage[(m0 + r) * LD + n0 + cc], v0, v1); });
      }
    }
    __syncthreads();

    // ---- state copy for the next chunk, output rows to HBM
    Sacc.pairs([&](int r, int cc, float &v0, float &v1) {
      if (std::is_same<E, f16>::value) nbad |= f16_out(v0) | f16_out(v1);
      st2(&sm.s[(wr * SWM + r) * LD + wc * SWN + cc], v0, v1);
    });
    if (emit) {
      I *og = static_cast<I *>(a.o);
      const I *ostage = reinterpret_cast<const I *>(sm.w);
      constexpr int EPV = 16 / sizeof(I);
      constexpr int VPR = D / EPV;
      for (int e = threadIdx.x; e < CH * VPR; e += NTHREADS) {
        const int r = e / VPR, cc = (e % VPR) * EPV;
        if (r < nvalid)
          *reinterpret_cast<uint4 *>(og + ((size_t)(tok0 + r) * H + h) * D + cc) =
              *reinterpret_cast<const uint4 *>(&ostage[r * LD + cc]);
      }
    }
  }

  if (nbad && a.status) atomicOr(a.status, 1);
  // ---- end-of-segment state
  float *dst = nullptr;
  if (a.pass == 0) {
    dst = (transition ? a.Mbuf : a.Ebuf) + sh_idx * DD;
  } else if (j == nseg - 1 && a.ST) {
    dst = a.ST + ((size_t)n * H + h) * DD;
  }
  if (dst) {
    const int m0 = wr * SWM, n0 = wc * SWN;
    Sacc.pairs([&](int r, int cc, float &v0, float &v1) {
      *reinterpret_cast<float2 *>(dst + (size_t)(m0 + r) * D + n0 + cc) = make_float2(v0, v1);
    });
  }
}

template <typename I, int D> static int launch_fwd(const FwdArgs &a, dim3 grid, cudaStream_t st) {
  using E = typename OpType<I>::T;
  const size_t smem = sizeof(FwdSmem<E, D>);
  static_assert(sizeof(FwdSmem<E, D>) <= 232448, "shared memory budget");
  auto kern = fwd_chunk_kernel<I, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  kern<<<grid, NTHREADS, smem, st>>>(a);
  return (int)cudaGetLastError();
}

int launch_fwd_chunk(const FwdArgs &a, bool is_bf16, int D, dim3 grid, cudaStream_t st) {
  if (is_bf16 && D == 128) return launch_fwd<bf16, 128>(a, grid, st);
  if (is_bf16 && D == 64) return launch_fwd<bf16, 64>(a, grid, st);
  if (!is_bf16 && D == 64) return launch_fwd<float, 64>(a, grid, st);
  return -1;
}

}  // namespace gdn
