// Chunked backward of the gated delta rule.
//
// The chunk graph of the forward (see fwd.cu) is differentiated by hand.  With
// dS the gradient w.r.t. a chunk's end state, per chunk:
//   Y     = K dS^T;   dUt = diag(cdec) Y + P^T dO
//   dS0   = gam_C dS + (diag(gam) dO)^T Q - dUt^T W           (reverse chain)
//   dQ    = diag(gam) dO S0 + dPm K,  dPm = diag(gp) tril_incl(dO Ut^T) diag(rgp)
//   dK    = diag(cdec) Ut dS + dPm^T Q + diag(beta) Ahat^T dW' + (dN + dN^T) K
//   dV    = X2^T dUt,  X2 = diag(gp) Ahat diag(beta rgp)  (the forward's bounded operand)
//   with dW' = diag(gam) dW = -diag(gam) dUt S0,
//   dAhat = (dW' K^T + Gamma * (dUt V^T)) diag(beta),  Gamma_ri = gp_r rgp_i (i <= r),
//   dT = -Ahat^T dAhat Ahat^T,  dN = strict_tril(diag(beta) dT).
// The last line forms dA and dA^T as one symmetric matrix multiplied with K
// once (onedev.kr FlashQLA talk summary, paragraph on SFU load, last sentence).
// Gate and beta gradients collect the row/column sums of the elementwise
// products listed in the local kernel and end with an in-chunk reverse cumsum.
//
// Kernels:
//   bwd_chain_kernel  one CTA per (segment, head): the serial reverse chain of
//                     dS, storing dS at every chunk end (pass 1), or the
//                     segment's start gradient / transition (pass 0) for the
//                     reverse sequence-parallel fix-up.
//   bwd_local_kernel  one CTA per (chunk, head): every local gradient, given
//                     the forward state at the chunk start and dS at its end.
#include "chunk_common.cuh"
#include "kernels.h"

namespace gdn {

// ============================================================== reverse chain
template <typename E, int D> struct ChainSmem {
  static constexpr int LD = D + Pad<E>::v;
  static constexpr int LC = CH + Pad<E>::v;
  static constexpr int LN = CH + 4;
  E q[CH * LD], k[CH * LD], dob[CH * LD], dog[CH * LD], w[CH * LD], du[CH * LD];
  E ds[D * LD];
  E p[CH * LC], x1[CH * LC];
  float nf[CH * LN];
  float g[CH], beta[CH];
  Gates gt;
  float ys[1152];
};

template <typename I, int D>
__global__ void __launch_bounds__(NTHREADS, 1) bwd_chain_kernel(BwdArgs a) {
  using E = typename OpType<I>::T;
  using SM = ChainSmem<E, D>;
  constexpr int LD = SM::LD, LC = SM::LC, LN = SM::LN;
  constexpr int SWM = D / 4, SWN = D / 2;
  extern __shared__ __align__(128) unsigned char smraw[];
  SM &sm = *reinterpret_cast<SM *>(smraw);

  const int s = blockIdx.x, h = blockIdx.y, role = blockIdx.z;
  // pass A of a call in which no segment needs the exact fix-up (status[2], set by the fix-up mode scan)
  if (a.pass == 0 && a.status && a.status[2] == 0) return;
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
  const int mode = bwd_start_mode(a.gsum, H, h, chunk0, cend, nchunks, j, nseg, window, &w);
  bool transition = false;
  if (a.pass == 0) {
    if (j == 0) return;
    int w2;
    if (bwd_start_mode(a.gsum, H, h, chunk0, cbeg, nchunks, j - 1, nseg, window, &w2) != START_FIXUP) return;
    if (role == 1) {
      if (mode != START_FIXUP) return;
      transition = true;
    }
  } else if (role != 0) {
    return;
  }
  const bool store = (a.pass == 1);
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  const int warp = threadIdx.x >> 5;
  const int wr = warp >> 1, wc = warp & 1;
  const I *qg = static_cast<const I *>(a.q);
  const I *kg = static_cast<const I *>(a.k);
  const I *dog = static_cast<const I *>(a.dO);
  const size_t DD = (size_t)D * D;
  const size_t sh_idx = (size_t)s * H + h;

  int clast = cend - 1;  // first chunk processed (reverse order)
  if (mode == START_WARMUP && !transition) clast = cend - 1 + w;

  auto issue_loads = [&](int c) {
    const long tok0 = bos + (long)c * CH;
    const int nvalid = min(CH, len - c * CH);
    load_tile<I, D>(sm.k, LD, kg, H, h, tok0, nvalid);
    if (!transition) {
      load_tile<I, D>(sm.q, LD, qg, H, h, tok0, nvalid);
      load_tile<I, D>(sm.dob, LD, dog, H, h, tok0, nvalid);
    }
    load_scalars(sm.g, a.g, H, h, tok0, nvalid, 0);
    load_scalars(sm.beta, a.beta, H, h, tok0, nvalid, 64);
    cp_async_commit();
  };
  issue_loads(clast);

  Acc<SWM, SWN> dS;
  bool nbad = false;  // numeric guard: an fp16 operand out of range
  {
    const float *src = nullptr;
    if (!transition) {
      if (mode == START_INIT) src = a.dST ? a.dST + ((size_t)n * H + h) * DD : nullptr;
      else if (mode == START_FIXUP && a.pass != 0) src = a.dSend + sh_idx * DD;
    }
    const int m0 = wr * SWM, n0 = wc * SWN;
    dS.pairs([&](int r, int c, float &v0, float &v1) {
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
      st2(&sm.ds[row * LD + col], v0, v1);
    });
  }

  for (int c = clast; c >= cbeg; --c) {
    cp_async_wait_all();
    __syncthreads();
    if (store && c < cend) {
      E *dst = static_cast<E *>(a.dstates) + ((size_t)(chunk0 + c) * H + h) * DD;
      constexpr int EPV = 16 / sizeof(E);
      for (int e = threadIdx.x; e < D * D / EPV; e += NTHREADS) {
        const int r = e / (D / EPV), cc = (e % (D / EPV)) * EPV;
        *reinterpret_cast<uint4 *>(dst + (size_t)r * D + cc) = *reinterpret_cast<const uint4 *>(&sm.ds[r * LD + cc]);
      }
    }
    nbad |= prep_rows<I, E, D>(sm.k, LD, 1.f, l2, nullptr);
    if (!transition) {
      nbad |= prep_rows<I, E, D>(sm.q, LD, a.scale, l2, nullptr);
      nbad |= prep_rows<I, E, D>(sm.dob, LD, 1.f, false, nullptr);
    }
    if (warp == 0) gate_prefix(sm.g, sm.gt);
    __syncthreads();

    // N (warps 0-3), P (warps 4-7), diag(gam) dO
    if (!transition) {
      for (int e = threadIdx.x; e < CH * D; e += NTHREADS) {
        const int r = e / D, cc = e % D;
        sm.dog[r * LD + cc] = fromf<E>(tof(sm.dob[r * LD + cc]) * sm.gt.gam[r]);
      }
    }
    if (warp < 4 || !transition) {
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
      st2(&sm.x1[r * LC + c], a0 * sm.beta[c], a1 * sm.beta[c + 1]);
    });

    // W = diag(gam) X1 K  (all warps: 64 x D as 4 x 2 tiles of 16 x D/2)
    {
      Acc<16, SWN> acc;
      acc.zero();
      const int m0 = wr * 16, n0 = wc * SWN;
      warp_mma<16, SWN, false, true>(acc, sm.x1, LC, sm.k, LD, m0, n0, CH);
      acc.pairs([&](int r, int cc, float &v0, float &v1) {
        const float gm = sm.gt.gam[m0 + r];
        st2(&sm.w[(m0 + r) * LD + n0 + cc], v0 * gm, v1 * gm);
      });
    }
    // dUt = diag(cdec) K dS^T + P^T dO ; stored negated
    {
      Acc<16, SWN> acc;
      acc.zero();
      const int m0 = wr * 16, n0 = wc * SWN;
      warp_mma<16, SWN, false, false>(acc, sm.k, LD, sm.ds, LD, m0, n0, D);
      acc.each([&](int r, int cc, float &v) { v *= sm.gt.cdec[m0 + r]; });
      if (!transition) warp_mma<16, SWN, true, true>(acc, sm.p, LC, sm.dob, LD, m0, n0, CH);
      acc.pairs([&](int r, int cc, float &v0, float &v1) { st2(&sm.du[(m0 + r) * LD + n0 + cc], -v0, -v1); });
    }
    __syncthreads();

    // dS <- gam_C dS + (diag(gam) dO)^T Q + (-dUt)^T W
    {
      const float gC = sm.gt.gamC;
      dS.each([&](int r, int cc, float &v) { v *= gC; });
      const int m0 = wr * SWM, n0 = wc * SWN;
      if (!transition) warp_mma<SWM, SWN, true, true>(dS, sm.dog, LD, sm.q, LD, m0, n0, CH);
      warp_mma<SWM, SWN, true, true>(dS, sm.du, LD, sm.w, LD, m0, n0, CH);
    }
    __syncthreads();
    if (c - 1 >= cbeg) issue_loads(c - 1);  // K, Q, dO, g, beta tiles are free now
    dS.pairs([&](int r, int cc, float &v0, float &v1) {
      if (std::is_same<E, f16>::value) nbad |= f16_out(v0) | f16_out(v1);
      st2(&sm.ds[(wr * SWM + r) * LD + wc * SWN + cc], v0, v1);
    });
  }
  if (nbad && a.status) atomicOr(a.status, 1);

  float *dst = nullptr;
  if (a.pass == 0) dst = (transition ? a.Rbuf : a.Fbuf) + sh_idx * DD;
  else if (j == 0 && a.dS0) dst = a.dS0 + ((size_t)n * H + h) * DD;
  if (dst) {
    const int m0 = wr * SWM, n0 = wc * SWN;
    dS.pairs([&](int r, int cc, float &v0, float &v1) {
      *reinterpret_cast<float2 *>(dst + (size_t)(m0 + r) * D + n0 + cc) = make_float2(v0, v1);
    });
  }
}

// ============================================================ local gradients
template <typename E, int D> struct LocalSmem {
  static constexpr int LD = D + Pad<E>::v;
  static constexpr int LC = CH + Pad<E>::v;
  static constexpr int LN = CH + 4;
  E q[CH * LD], k[CH * LD], v[CH * LD], dob[CH * LD];
  E s0[D * LD];
  E ds[D * LD];  // dS, later reused for dUt
  E ut[CH * LD], w[CH * LD];
  E p[CH * LC], x1[CH * LC], x2[CH * LC];  // p later holds dPm, then Sigma; x2 later holds Ahat
  float nf[CH * LN];
  float g[CH], beta[CH], nq[CH], nk[CH];
  Gates gt;
  float ys[1152];
  float part[18][CH];   // gate-gradient partials (see the final sum)
  float bpart[6][CH];   // beta-gradient partials
  float rdot[2][CH];    // row dots for the normalisation Jacobians
  float red[NWARPS];
};

template <typename I, int D>
__global__ void __launch_bounds__(NTHREADS, 1) bwd_local_kernel(BwdArgs a) {
  using E = typename OpType<I>::T;
  using SM = LocalSmem<E, D>;
  constexpr int LD = SM::LD, LC = SM::LC, LN = SM::LN;
  constexpr int WN = D / 2;
  extern __shared__ __align__(128) unsigned char smraw[];
  SM &sm = *reinterpret_cast<SM *>(smraw);
  const int gc = blockIdx.x, h = blockIdx.y;
  const int H = a.H;
  const int n = a.plan.chunk_seq[gc];
  if (n < 0) return;
  const int lc = gc - a.plan.seq_chunk0[n];
  const int len = a.plan.seq_len[n];
  const long tok0 = (long)a.plan.seq_bos[n] + (long)lc * CH;
  const int nvalid = min(CH, len - lc * CH);
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = warp >> 1, wc = warp & 1;
  const size_t DD = (size_t)D * D;
  const size_t st_idx = ((size_t)gc * H + h) * DD;

  // ---- loads
  load_tile<I, D>(sm.q, LD, static_cast<const I *>(a.q), H, h, tok0, nvalid);
  load_tile<I, D>(sm.k, LD, static_cast<const I *>(a.k), H, h, tok0, nvalid);
  load_tile<I, D>(sm.v, LD, static_cast<const I *>(a.v), H, h, tok0, nvalid);
  load_tile<I, D>(sm.dob, LD, static_cast<const I *>(a.dO), H, h, tok0, nvalid);
  load_scalars(sm.g, a.g, H, h, tok0, nvalid, 0);
  load_scalars(sm.beta, a.beta, H, h, tok0, nvalid, 64);
  {
    constexpr int EPV = 16 / sizeof(E);
    const E *s0g = static_cast<const E *>(a.states) + st_idx;
    const E *dsg = static_cast<const E *>(a.dstates) + st_idx;
    for (int e = threadIdx.x; e < D * D / EPV; e += NTHREADS) {
      const int r = e / (D / EPV), cc = (e % (D / EPV)) * EPV;
      cp_async16(&sm.s0[r * LD + cc], s0g + (size_t)r * D + cc, true);
      cp_async16(&sm.ds[r * LD + cc], dsg + (size_t)r * D + cc, true);
    }
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  prep_rows<I, E, D>(sm.k, LD, 1.f, l2, sm.nk);
  prep_rows<I, E, D>(sm.q, LD, a.scale, l2, sm.nq);
  prep_rows<I, E, D>(sm.v, LD, 1.f, false, nullptr);
  prep_rows<I, E, D>(sm.dob, LD, 1.f, false, nullptr);
  if (warp == 0) gate_prefix(sm.g, sm.gt);
  __syncthreads();

  // ---- N, P
  {
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
  wy_inverse<std::is_same<E, float>::value, true>(sm.nf, LN, sm.beta, sm.ys,
                                                    [&](int r, int c, float a0, float a1) {
    const float b0 = sm.beta[c], b1 = sm.beta[c + 1];
    st2(&sm.x1[r * LC + c], a0 * b0, a1 * b1);
    st2(&sm.x2[r * LC + c], c <= r ? a0 * b0 * gratio(sm.gt, r, c) : 0.f,
        c + 1 <= r ? a1 * b1 * gratio(sm.gt, r, c + 1) : 0.f);
  });

  const int m0 = wr * 16, n0 = wc * WN;  // 64 x D outputs: 4 x 2 warps of 16 x D/2
  // ---- -W  and  Ut = U - W S0^T
  {
    Acc<16, WN> acc;
    acc.zero();
    warp_mma<16, WN, false, true>(acc, sm.x1, LC, sm.k, LD, m0, n0, CH);
    acc.pairs([&](int r, int cc, float &v0, float &v1) {
      const float gm = -sm.gt.gam[m0 + r];
      st2(&sm.w[(m0 + r) * LD + n0 + cc], v0 * gm, v1 * gm);
    });
  }
  __syncthreads();
  {
    Acc<16, WN> acc;
    acc.zero();
    warp_mma<16, WN, false, true>(acc, sm.x2, LC, sm.v, LD, m0, n0, CH);
    warp_mma<16, WN, false, false>(acc, sm.w, LD, sm.s0, LD, m0, n0, D);
    acc.pairs([&](int r, int cc, float &v0, float &v1) { st2(&sm.ut[(m0 + r) * LD + n0 + cc], v0, v1); });
  }
  __syncthreads();

  // ---- Y = K dS^T: y-terms <Ut, Y>; dUt = diag(cdec) Y + P^T dO
  Acc<16, WN> dU;
  {
    dU.zero();
    warp_mma<16, WN, false, false>(dU, sm.k, LD, sm.ds, LD, m0, n0, D);
    float ry[2] = {0.f, 0.f};
    dU.each([&](int r, int cc, float &v) { ry[r >> 3] += v * tof(sm.ut[(m0 + r) * LD + n0 + cc]); });
    dU.each([&](int r, int cc, float &v) { v *= sm.gt.cdec[m0 + r]; });
    warp_mma<16, WN, true, true>(dU, sm.p, LC, sm.dob, LD, m0, n0, CH);
#pragma unroll
    for (int t = 0; t < 2; ++t) ry[t] = quad_sum(ry[t]);
    if ((lane & 3) == 0) {
      const int r = m0 + (lane >> 2);
      sm.part[0 + wc][r] = ry[0];
      sm.part[0 + wc][r + 8] = ry[1];
    }
  }
  // dK accumulator (kept in registers): diag(cdec) Ut dS
  Acc<16, WN> dK;
  dK.zero();
  warp_mma<16, WN, false, true>(dK, sm.ut, LD, sm.ds, LD, m0, n0, D);
  dK.each([&](int r, int cc, float &v) { v *= sm.gt.cdec[m0 + r]; });
  // gam_C <dS, S0>
  {
    float acc = 0.f;
    for (int e = threadIdx.x; e < D * D; e += NTHREADS) {
      const int r = e / D, cc = e % D;
      acc += tof(sm.ds[r * LD + cc]) * tof(sm.s0[r * LD + cc]);
    }
    acc = warp_sum(acc);
    if (lane == 0) sm.red[warp] = acc;
  }
  __syncthreads();  // everyone done with sm.ds (dS)
  E *du = sm.ds;   // dUt   (CH x LD; dS is no longer needed)
  E *dw = sm.dob;  // dW' = -diag(gam) dUt S0 (written after the last read of dO)
  dU.pairs([&](int r, int cc, float &v0, float &v1) { st2(&du[(m0 + r) * LD + n0 + cc], v0, v1); });
  // ---- dP = dO Ut^T  ->  Z = dP * P sums, dPm (written over P, element by element)
  E *dpm = sm.p;
  {
    Acc<16, 32> acc;
    acc.zero();
    const int pm0 = wr * 16, pn0 = wc * 32;
    warp_mma<16, 32, false, false>(acc, sm.dob, LD, sm.ut, LD, pm0, pn0, D);
    float rs[2] = {0.f, 0.f};
    float cs[4][2];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) cs[jj][0] = cs[jj][1] = 0.f;
    acc.each([&](int r, int cc, float &v) {
      const int row = pm0 + r, col = pn0 + cc;
      const float pv = tof(sm.p[row * LC + col]);
      const float z = v * pv;
      rs[r >> 3] += z;
      cs[cc >> 3][cc & 1] += z;
      dpm[row * LC + col] = fromf<E>(col <= row ? v * gratio(sm.gt, row, col) : 0.f);
    });
#pragma unroll
    for (int t = 0; t < 2; ++t) rs[t] = quad_sum(rs[t]);
    if ((lane & 3) == 0) {
      sm.part[4 + wc][pm0 + (lane >> 2)] = rs[0];
      sm.part[4 + wc][pm0 + (lane >> 2) + 8] = rs[1];
    }
    // column sums: reduce over the 8 row-lanes sharing lane % 4
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float x = cs[jj][t];
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        if (lane < 4) sm.part[6 + wr][pn0 + 8 * jj + 2 * lane + t] = x;
      }
  }
  __syncthreads();

  // ---- dQ = diag(gam) dO S0 + dPm K
  {
    Acc<16, WN> acc;
    acc.zero();
    warp_mma<16, WN, false, true>(acc, sm.dob, LD, sm.s0, LD, m0, n0, D);
    float rq[2] = {0.f, 0.f};
    acc.each([&](int r, int cc, float &v) {
      v *= sm.gt.gam[m0 + r];
      rq[r >> 3] += v * tof(sm.q[(m0 + r) * LD + n0 + cc]);
    });
    warp_mma<16, WN, false, true>(acc, dpm, LC, sm.k, LD, m0, n0, CH);
    float rj[2] = {0.f, 0.f};
    acc.each([&](int r, int cc, float &v) { rj[r >> 3] += v * tof(sm.q[(m0 + r) * LD + n0 + cc]); });
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      rq[t] = quad_sum(rq[t]);
      rj[t] = quad_sum(rj[t]);
    }
    if ((lane & 3) == 0) {
      const int r = m0 + (lane >> 2);
      sm.part[10 + wc][r] = rq[0];
      sm.part[10 + wc][r + 8] = rq[1];
      sm.rdot[wc][r] = rj[0];
      sm.rdot[wc][r + 8] = rj[1];
    }
    __syncthreads();
    // dq = scale * dq^ (no norm), or (scale dq^ - Q^ (Q^ . dq^) / scale) / |q|
    I *dqg = static_cast<I *>(a.dq);
    acc.pairs([&](int r, int cc, float &v0, float &v1) {
      const int row = m0 + r;
      if (row >= nvalid) return;
      float o0, o1;
      if (l2) {
        const float dot = sm.rdot[0][row] + sm.rdot[1][row];
        const float inv = 1.f / sm.nq[row];
        o0 = (a.scale * v0 - tof(sm.q[row * LD + n0 + cc]) * dot / a.scale) * inv;
        o1 = (a.scale * v1 - tof(sm.q[row * LD + n0 + cc + 1]) * dot / a.scale) * inv;
      } else {
        o0 = a.scale * v0;
        o1 = a.scale * v1;
      }
      st2(dqg + ((size_t)(tok0 + row) * H + h) * D + n0 + cc, o0, o1);
    });
  }
  // ---- dW' = -diag(gam) dUt S0
  {
    Acc<16, WN> acc;
    acc.zero();
    warp_mma<16, WN, false, true>(acc, du, LD, sm.s0, LD, m0, n0, D);
    acc.pairs([&](int r, int cc, float &v0, float &v1) {
      const float gm = -sm.gt.gam[m0 + r];
      st2(&dw[(m0 + r) * LD + n0 + cc], v0 * gm, v1 * gm);
    });
  }
  __syncthreads();
  // ---- dK += dPm^T Q + X1^T dW'
  warp_mma<16, WN, true, true>(dK, dpm, LC, sm.q, LD, m0, n0, CH);
  warp_mma<16, WN, true, true>(dK, sm.x1, LC, dw, LD, m0, n0, CH);
  // ---- dV = X2^T dUt
  {
    Acc<16, WN> acc;
    acc.zero();
    warp_mma<16, WN, true, true>(acc, sm.x2, LC, du, LD, m0, n0, CH);
    I *dvg = static_cast<I *>(a.dv);
    acc.pairs([&](int r, int cc, float &v0, float &v1) {
      const int row = m0 + r;
      if (row < nvalid) st2(dvg + ((size_t)(tok0 + row) * H + h) * D + n0 + cc, v0, v1);
    });
  }
  // ---- dAhat = (dW' K^T + Gamma * (dUt V^T)) diag(beta); beta column terms
  {
    Acc<16, 32> a1, a2;
    a1.zero();
    a2.zero();
    const int pm0 = wr * 16, pn0 = wc * 32;
    warp_mma<16, 32, false, false>(a1, dw, LD, sm.k, LD, pm0, pn0, D);
    warp_mma<16, 32, false, false>(a2, du, LD, sm.v, LD, pm0, pn0, D);
    float cs[4][2], xc[4][2], rwx[2] = {0.f, 0.f};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) cs[jj][0] = cs[jj][1] = xc[jj][0] = xc[jj][1] = 0.f;
    // element (r, i): a1 = <dW'_r, k_i>, a2 = <dUt_r, v_i>; the V term carries
    // Gamma_ri = gamma_r / gamma_i <= 1 for i <= r (entries above the diagonal do not
    // reach the strictly lower part of dT and are dropped).  Gate terms: <dW_r, W_r> =
    // rowsum_r(beta Ahat a1) and the row / column sums of X2 * a2 = beta Ahat Gamma a2 over the
    // strictly lower triangle (a diagonal ratio does not depend on the gates; leaving it out of both
    // sums avoids a difference of two large, differently rounded numbers under strong decay)
    {
      const int lr = lane >> 2, lcc = 2 * (lane & 3);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = pm0 + lr + 8 * (e >> 1), col = pn0 + 8 * jj + lcc + (e & 1);
          const float ah = ahat_at(sm.nf, LN, row, col);
          const float x1 = a1.c[0][jj][e];
          const float x2 = col <= row ? a2.c[0][jj][e] * gratio(sm.gt, row, col) : 0.f;
          const float xo = col < row ? sm.beta[col] * ah * x2 : 0.f;
          rwx[e >> 1] += sm.beta[col] * ah * x1 + xo;
          xc[jj][e & 1] += xo;
          cs[jj][e & 1] += ah * (x1 + x2);
          a1.c[0][jj][e] = sm.beta[col] * (x1 + x2);
        }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) rwx[t] = quad_sum(rwx[t]);
    if ((lane & 3) == 0) {
      sm.part[2 + wc][pm0 + (lane >> 2)] = rwx[0];
      sm.part[2 + wc][pm0 + (lane >> 2) + 8] = rwx[1];
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float x = xc[jj][t];
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        if (lane < 4) sm.part[14 + wr][pn0 + 8 * jj + 2 * lane + t] = x;
      }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float x = cs[jj][t];
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        if (lane < 4) sm.bpart[wr][pn0 + 8 * jj + 2 * lane + t] = x;
      }
    // dAhat (E) into the W tile region (W no longer needed)
    E *dA = sm.w;
    a1.pairs([&](int r, int cc, float &v0, float &v1) { st2(&dA[(pm0 + r) * LC + pn0 + cc], v0, v1); });
  }
  __syncthreads();
  // ---- Y1 = Ahat^T dAhat ; dT = -Y1 Ahat^T ; Sigma = dN + dN^T
  E *dA = sm.w;   // W no longer needed
  E *Y1 = sm.ut;  // Ut no longer needed
  E *Sig = sm.p;  // dPm no longer needed
  E *ah = sm.x2;  // X2 no longer needed
  for (int e = threadIdx.x; e < CH * CH; e += NTHREADS) {
    const int r = e / CH, i = e % CH;
    ah[r * LC + i] = fromf<E>(ahat_at(sm.nf, LN, r, i));
  }
  __syncthreads();
  {
    Acc<16, 32> acc;
    acc.zero();
    const int pm0 = wr * 16, pn0 = wc * 32;
    warp_mma<16, 32, true, true>(acc, ah, LC, dA, LC, pm0, pn0, CH);
    acc.pairs([&](int r, int cc, float &v0, float &v1) { st2(&Y1[(pm0 + r) * LC + pn0 + cc], v0, v1); });
  }
  __syncthreads();
  {
    Acc<16, 32> acc;
    acc.zero();
    const int pm0 = wr * 16, pn0 = wc * 32;
    warp_mma<16, 32, false, false>(acc, Y1, LC, ah, LC, pm0, pn0, CH);
    float rb[2] = {0.f, 0.f};
    acc.each([&](int r, int cc, float &v) {
      const int row = pm0 + r, col = pn0 + cc;
      const float dT = -v;
      if (col < row) {
        rb[r >> 3] += dT * sm.nf[row * LN + col];
        const float dn = sm.beta[row] * dT;
        Sig[row * LC + col] = fromf<E>(dn);
        Sig[col * LC + row] = fromf<E>(dn);
      } else if (col == row) {
        Sig[row * LC + col] = fromf<E>(0.f);
      }
    });
#pragma unroll
    for (int t = 0; t < 2; ++t) rb[t] = quad_sum(rb[t]);
    if ((lane & 3) == 0) {
      sm.bpart[4 + wc][pm0 + (lane >> 2)] = rb[0];
      sm.bpart[4 + wc][pm0 + (lane >> 2) + 8] = rb[1];
    }
  }
  __syncthreads();
  // ---- dK += Sigma K ; normalisation Jacobian ; store
  warp_mma<16, WN, false, true>(dK, Sig, LC, sm.k, LD, m0, n0, CH);
  {
    float rk[2] = {0.f, 0.f};
    dK.each([&](int r, int cc, float &v) { rk[r >> 3] += v * tof(sm.k[(m0 + r) * LD + n0 + cc]); });
#pragma unroll
    for (int t = 0; t < 2; ++t) rk[t] = quad_sum(rk[t]);
    if ((lane & 3) == 0) {
      sm.rdot[wc][m0 + (lane >> 2)] = rk[0];
      sm.rdot[wc][m0 + (lane >> 2) + 8] = rk[1];
    }
  }
  __syncthreads();
  {
    I *dkg = static_cast<I *>(a.dk);
    dK.pairs([&](int r, int cc, float &v0, float &v1) {
      const int row = m0 + r;
      if (row >= nvalid) return;
      float o0 = v0, o1 = v1;
      if (l2) {
        const float dot = sm.rdot[0][row] + sm.rdot[1][row];
        const float inv = 1.f / sm.nk[row];
        o0 = (v0 - tof(sm.k[row * LD + n0 + cc]) * dot) * inv;
        o1 = (v1 - tof(sm.k[row * LD + n0 + cc + 1]) * dot) * inv;
      }
      st2(dkg + ((size_t)(tok0 + row) * H + h) * D + n0 + cc, o0, o1);
    });
  }
  // ---- gate and beta gradients
  if (warp == 0) {
    // dg_t = sum_{r >= t} dG_r + gam_C <dS, S0> + sum_{r < t} y_r (the state terms y_r = cdec_r <Ut_r, Y_r>
    // depend on g_t only for r < t): a reverse inclusive scan of dG and a forward exclusive scan of y
    float dGv[2], yv[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r = lane + 32 * t;
      yv[t] = sm.gt.cdec[r] * (sm.part[0][r] + sm.part[1][r]);
      float d = sm.part[2][r] + sm.part[3][r];                                     // <dW, W> + X2 * M2 rows
      d += sm.part[4][r] + sm.part[5][r];                                          // row sums of dP * P
      d -= sm.part[6][r] + sm.part[7][r] + sm.part[8][r] + sm.part[9][r];          // column sums
      d += sm.part[10][r] + sm.part[11][r];                                        // gam <dO, S0 q>
      d -= sm.part[14][r] + sm.part[15][r] + sm.part[16][r] + sm.part[17][r];      // X2 * M2 columns
      dGv[t] = d;
    }
    float red = 0.f;
    for (int i = 0; i < NWARPS; ++i) red += sm.red[i];
    float hi = dGv[1], lo = dGv[0], ylo = yv[0], yhi = yv[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float yh = __shfl_down_sync(0xffffffffu, hi, o), yl = __shfl_down_sync(0xffffffffu, lo, o);
      const float fl = __shfl_up_sync(0xffffffffu, ylo, o), fh = __shfl_up_sync(0xffffffffu, yhi, o);
      if (lane + o < 32) {
        hi += yh;
        lo += yl;
      }
      if (lane >= o) {
        ylo += fl;
        yhi += fh;
      }
    }
    lo += __shfl_sync(0xffffffffu, hi, 0);
    yhi += __shfl_sync(0xffffffffu, ylo, 31);
    const float base = sm.gt.gamC * red;
    lo += base + (ylo - yv[0]);
    hi += base + (yhi - yv[1]);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r = lane + 32 * t;
      if (r < nvalid) {
        a.dg[(size_t)(tok0 + r) * H + h] = t ? hi : lo;
        const float db = sm.bpart[0][r] + sm.bpart[1][r] + sm.bpart[2][r] + sm.bpart[3][r] + sm.bpart[4][r] +
                         sm.bpart[5][r];
        a.dbeta[(size_t)(tok0 + r) * H + h] = db;
      }
    }
  }
}

// ================================================================== launchers
template <typename I, int D> static int launch_chain(const BwdArgs &a, dim3 grid, cudaStream_t st) {
  using E = typename OpType<I>::T;
  const size_t smem = sizeof(ChainSmem<E, D>);
  static_assert(sizeof(ChainSmem<E, D>) <= 232448, "shared memory budget");
  auto kern = bwd_chain_kernel<I, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  kern<<<grid, NTHREADS, smem, st>>>(a);
  return (int)cudaGetLastError();
}
template <typename I, int D> static int launch_local(const BwdArgs &a, int CH_max, cudaStream_t st) {
  using E = typename OpType<I>::T;
  const size_t smem = sizeof(LocalSmem<E, D>);
  static_assert(sizeof(LocalSmem<E, D>) <= 232448, "shared memory budget");
  auto kern = bwd_local_kernel<I, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  kern<<<dim3(CH_max, a.H), NTHREADS, smem, st>>>(a);
  return (int)cudaGetLastError();
}

int launch_bwd_chain(const BwdArgs &a, bool is_bf16, int D, dim3 grid, cudaStream_t st) {
  if (is_bf16 && D == 128) return launch_chain<bf16, 128>(a, grid, st);
  if (is_bf16 && D == 64) return launch_chain<bf16, 64>(a, grid, st);
  if (!is_bf16 && D == 64) return launch_chain<float, 64>(a, grid, st);
  return -1;
}
int launch_bwd_local(const BwdArgs &a, bool is_bf16, int D, int CH_max, cudaStream_t st) {
  if (CH_max == 0) return 0;
  // bf16 with d = 128 reaches this kernel only for a call without tokens (its local gradients run on the
  // tensor cores otherwise), where there is no chunk to differentiate
  if (is_bf16 && D == 128) return 0;
  if (is_bf16 && D == 64) return launch_local<bf16, 64>(a, CH_max, st);
  if (!is_bf16 && D == 64) return launch_local<float, 64>(a, CH_max, st);
  return -1;
}

}  // namespace gdn
