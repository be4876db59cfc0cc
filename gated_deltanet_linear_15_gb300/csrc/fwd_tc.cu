// Blackwell-native fused forward (bf16 inputs, d = 128): TMA tile loads,
// tcgen05.mma with every accumulator in tensor memory (TMEM), the recurrent
// state resident in TMEM for the whole segment.
//
// Every chunk product is an M = 128 MMA with the feature dimension on the
// TMEM lanes (transposed where that is what puts d = 128 on M):
//   [K; Q] K^T     -> N = strict_tril(K K^T) (rows 0-63), Q K^T (rows 64-127)
//   W^T = K^T X1^T, U^T = V^T X2^T      X1 = Ahat diag(beta), X2 = diag(gp) Ahat diag(beta rgp)
//   Ut^T = U^T - S0 W^T (negated-A MMA accumulating on U^T),   Oi^T = S0 Q^T
//   S   = gam_C S0 + (Ut^T diag(cdec)) K    (K as the MN-major operand)
//   Oa^T = Ut^T P^T                         P = diag(gp) tril_incl(Q K^T) diag(rgp)
//   O^T = Oi^T diag(gam) + Oa^T             (combined at read-out)
// with W^T's columns scaled by gam and a cdec-scaled copy of Ut^T made at read-out, and
// Ahat = (I + diag(beta) N)^{-1} computed on CUDA cores in fp32 (onedev.kr
// FlashQLA talk summary, paragraph on the WY representation for the four
// steps; paragraph on SFU load for pulling the diagonal gamma scaling out of
// the inverse).  Operands are fp16 in 128-byte-swizzled shared memory (see
// umma.cuh); the state is kept in fp32 in TMEM and copied to fp16 once per
// chunk as the operand of the next products.
//
// One CTA of 512 threads per (segment, head); thread 0 issues TMA and MMA,
// all 16 warps read TMEM (warp w reaches lanes 32 (w % 4)..; the four warps of
// a lane quarter split the columns) and do the CUDA-core work.  Inputs of chunk c+1 are loaded by TMA while chunk c is computed, and
// normalised in place (they need no gates) while chunk c's last two MMA groups
// run.
#include "chunk_common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {

using namespace umma;

namespace {

constexpr int D = 128;
constexpr int HT = 8192;  // one 64 x 64 fp16 half-tile, 128B-swizzled
constexpr int FT = 512;   // worker threads (16 warps); warp 16 is the producer
constexpr int FWARPS = FT / 32;

// TMEM columns
constexpr uint32_t TM_S = 0, TM_KQ = 128, TM_W = 192, TM_U = 256, TM_O = 320, TM_OA = 384, TM_COLS = 512;

struct __align__(1024) TcSmem {
  // input ring, 2 stages: [K0 | Q0 | K1 | Q1 | V0 | V1] half-tiles (0/1 = feature block)
  uint8_t ring[2][6 * HT];
  uint8_t uc[2 * HT];   // Ut^T diag(cdec) (K-major A, rows = d_v)
  uint8_t x1[HT], x2[HT], p[HT];
  uint8_t wu[2 * HT];   // W^T (MN-major B, rows = d_k), later Ut^T (K-major A, rows = d_v), then O staging
  uint8_t s0[4 * HT];   // S0 fp16 (K-major A: rows = d_v, two k-blocks of 128 rows)
  uint8_t ah[HT];       // Ahat fp16 (row-major, swizzled), staged for the saved-context store
  float nf[CH * (CH + 4)];
  float g[2][CH], beta[2][CH];  // per ring stage
  Gates gt[2];  // per ring stage; the next chunk's gates are computed during this chunk
  float ys[1152];
  uint64_t bar_tma[2];
  uint64_t bar_mma;
  uint64_t bar_kq;  // MMA 1 ([K; Q] K^T) of a chunk, issued right after the previous chunk's MMA 4
  uint32_t tmem_base;
};

constexpr int LN = CH + 4;

__device__ __forceinline__ uint32_t u32(const void *p) { return smem_u32(p); }

// store 8 fp32 values as one 16-byte fp16 chunk
__device__ __forceinline__ void st_chunk_f16(uint8_t *dst, const float *v) {
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<uint4 *>(h);
}

}  // namespace

// byte offset of the 16-byte chunk holding columns [cb, cb + 8) of row r in a swizzled [rows][64] tile
__device__ __forceinline__ uint32_t chunk_off(int r, int cb) { return r * 128 + ((((cb & 63) >> 3) ^ (r & 7)) << 4); }

__global__ void __launch_bounds__(FT + 32, 1)
    fwd_tc_kernel(FwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmw,
                  const __grid_constant__ CUtensorMap tms, const __grid_constant__ CUtensorMap tmt,
                  const __grid_constant__ CUtensorMap tm3) {
  extern __shared__ unsigned char smraw[];
  TcSmem &sm = *reinterpret_cast<TcSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  pdl_trigger();
  pdl_wait();

  const int s = blockIdx.x, h = blockIdx.y, role = blockIdx.z;
  // pass A of a call in which no segment needs the exact fix-up (status[1], set after the gate scan)
  if (a.pass == 0 && a.status && a.status[1] == 0) return;
  const int H = a.H;
  const int n = a.plan.seg_seq[s];
  if (n < 0) return;
  const int j = s - a.plan.seq_seg0[n], nseg = a.plan.seq_nseg[n];
  const int len = a.plan.seq_len[n], chunk0 = a.plan.seq_chunk0[n];
  const int bos = a.plan.seq_bos[n];
  const int nchunks = (len + CH - 1) / CH;
  const int cbeg = j * a.Lseg, cend = min(cbeg + a.Lseg, nchunks);
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
  if (a.flags & kFlagDebugWaitTimeout) {  // test hook: an expiring bounded wait, then return
    __shared__ uint64_t dbg_bar;
    if (threadIdx.x == 0) debug_expire_wait(&dbg_bar, a.status, 4);
    return;
  }
  const bool outputs = (a.pass == 1);
  const bool need_v = !transition;
  // chunk-start states and the chunk context tiles (X1, X2, Ahat, P, N, scaled W^T, Ut^T) leave shared
  // memory by TMA stores issued by thread 0 (N from registers); a pass with o == NULL computes P but
  // no output
  const bool save_states = a.pass != 0 && a.states != nullptr;
  const bool save_wy = outputs && a.t64 != nullptr;
  const bool want_o = outputs && a.o != nullptr;
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2;                      // column group 0..3 within a lane quarter
  const int row = ((warp & 3) << 5) | lane;      // TMEM lane this thread reads
  const size_t DD = (size_t)D * D;
  const size_t sh_idx = (size_t)s * H + h;
  int cfirst = cbeg;
  if (mode == START_WARMUP && !transition) cfirst = cbeg - w;

  // ---------------------------------------------------------------- set-up
  if (tid == 0) {
    mbar_init(u32(&sm.bar_tma[0]), 1);
    mbar_init(u32(&sm.bar_tma[1]), 1);
    mbar_init(u32(&sm.bar_mma), 1);
    mbar_init(u32(&sm.bar_kq), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmq);
    if (save_wy) {
      tma_prefetch_desc(&tmw);
      tma_prefetch_desc(&tmt);
      tma_prefetch_desc(&tm3);
    }
    if (save_states) tma_prefetch_desc(&tms);
  }
  if (warp == 0) {
    tmem_alloc(u32(&sm.tmem_base), TM_COLS);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tm = sm.tmem_base;
  const uint32_t tm_lane = (uint32_t)((warp & 3) * 32) << 16;

  auto issue_tma = [&](int c, int stage) {
    const int tok0 = bos + c * CH;
    const bool wq = outputs && c >= cbeg;
    const uint32_t bytes = (2 + (wq ? 2 : 0) + (need_v ? 2 : 0)) * HT;
    const uint32_t bar = u32(&sm.bar_tma[stage]);
    uint8_t *st = sm.ring[stage];
    mbar_expect_tx(bar, bytes);
    tma_load_3d(u32(st + 0 * HT), &tmk, 0, h, tok0, bar);
    tma_load_3d(u32(st + 2 * HT), &tmk, 64, h, tok0, bar);
    if (wq) {
      tma_load_3d(u32(st + 1 * HT), &tmq, 0, h, tok0, bar);
      tma_load_3d(u32(st + 3 * HT), &tmq, 64, h, tok0, bar);
    }
    if (need_v) {
      tma_load_3d(u32(st + 4 * HT), &tmv, 0, h, tok0, bar);
      tma_load_3d(u32(st + 5 * HT), &tmv, 64, h, tok0, bar);
    }
  };
  auto issue_gb = [&](int c, int stage, bool with_g) {  // cp.async of (g and) beta for chunk c
    const int tok0 = bos + c * CH;
    const int nvalid = min(CH, len - c * CH);
    if (with_g) load_scalars(sm.g[stage], a.g, H, h, tok0, nvalid, 0);
    load_scalars(sm.beta[stage], a.beta, H, h, tok0, nvalid, 64);
    cp_async_commit();
  };
  if (tid == FT && cfirst < cend) issue_tma(cfirst, 0);
  if (cfirst < cend) issue_gb(cfirst, 0, true);

  // ---------------------------------------------------------------- initial state -> TMEM
  {
    const float *src = nullptr;
    if (!transition) {
      if (mode == START_INIT) src = a.S0 ? a.S0 + ((size_t)n * H + h) * DD : nullptr;
      else if (mode == START_FIXUP && a.pass != 0) src = a.Sstart + sh_idx * DD;
    }
    if (warp < FWARPS) {
      const int c0 = wg * 32;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int col = c0 + i;
        v[i] = src ? src[(size_t)row * D + col] : (transition && col == row ? 1.f : 0.f);
      }
      tmem_st32(tm + tm_lane + TM_S + c0, v);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();

  int *err = a.status;
  uint32_t mma_phase = 0, kq_phase = 0;
  bool failed = false;
  auto mma_wait = [&]() {
    const bool ok = mbar_wait(u32(&sm.bar_mma), mma_phase, err, 4);
    mma_phase ^= 1;
    fence_after();
    return ok;
  };
  // MMA 1: [K; Q] K^T of the chunk in ring stage `stg` -> TM_KQ (M = 128, N = 64, K = 128); thread 0
  auto issue_mma1 = [&](const uint8_t *stg) {
    const uint32_t idesc = idesc_f16(128, 64, false, false);
    const uint32_t base = u32(stg);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t koff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
      mma_f16(tm + TM_KQ, sdesc(base + koff, 16, 1024), sdesc(base + koff, 16, 1024), idesc, kk > 0);
    }
    mma_commit(u32(&sm.bar_kq));
  };

  // In-place operand preparation of one ring stage: bf16 -> fp16, L2 norm of the q/k rows (q also
  // scaled), rows >= nvalid zeroed.  prep_kq: thread t takes quarter-row t % 256 of K (t < 256) or
  // of Q: 32 features = four 16-byte chunks of one 128-byte swizzled row; the four quarters of a row
  // sit in adjacent lanes (two shuffles for the squared norm).  prep_v: eighth-row t of V.
  auto prep_kq = [&](uint8_t *st, int nvalid, bool with_q, float *nrm_out) {
    const bool isq = tid >= 256;
    if (isq && !with_q) return;
    const int r = (tid >> 2) & 63, qq = tid & 3;
    uint8_t *rowp = st + (isq ? HT : 0) + (qq >> 1) * 2 * HT + r * 128;
    const int ch0 = (qq & 1) * 4;
    uint32_t raw[16];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const uint4 q4 = *reinterpret_cast<const uint4 *>(rowp + (((ch0 + cc) ^ (r & 7)) * 16));
      raw[4 * cc] = q4.x;
      raw[4 * cc + 1] = q4.y;
      raw[4 * cc + 2] = q4.z;
      raw[4 * cc + 3] = q4.w;
    }
    float mul = isq ? a.scale : 1.f;
    if (l2) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float lo = __uint_as_float(raw[i] << 16), hi = __uint_as_float(raw[i] & 0xffff0000u);
        ss = fmaf(lo, lo, fmaf(hi, hi, ss));
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      const float rn = rsqrtf(ss + 1e-6f);
      mul *= rn;
      if (nrm_out && qq == 0) nrm_out[(isq ? CH : 0) + r] = rn;  // context: 1/|k|, 1/|q| per token
    } else if (nrm_out && qq == 0) {
      nrm_out[(isq ? CH : 0) + r] = 1.f;
    }
    if (r >= nvalid) mul = 0.f;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t y[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w = raw[4 * cc + i];
        const __half2 a2 = __floats2half2_rn(__uint_as_float(w << 16) * mul, __uint_as_float(w & 0xffff0000u) * mul);
        y[i] = *reinterpret_cast<const uint32_t *>(&a2);
      }
      *reinterpret_cast<uint4 *>(rowp + (((ch0 + cc) ^ (r & 7)) * 16)) = make_uint4(y[0], y[1], y[2], y[3]);
    }
  };
  auto prep_v = [&](uint8_t *st, int nvalid) {
    const int r = tid >> 3, part = tid & 7;
    uint8_t *rowp = st + 4 * HT + (part >> 2) * HT + r * 128;
    const float mul = r < nvalid ? 1.f : 0.f;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int chk = (part & 3) * 2 + cc;
      uint4 q4 = *reinterpret_cast<const uint4 *>(rowp + ((chk ^ (r & 7)) * 16));
      uint32_t *w = reinterpret_cast<uint32_t *>(&q4);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 a2 =
            __floats2half2_rn(__uint_as_float(w[i] << 16) * mul, __uint_as_float(w[i] & 0xffff0000u) * mul);
        w[i] = *reinterpret_cast<const uint32_t *>(&a2);
      }
      *reinterpret_cast<uint4 *>(rowp + ((chk ^ (r & 7)) * 16)) = q4;
    }
  };

  // Worker warps 0-15 do the read-outs and the CUDA-core work; lane 0 of warp 16 (the producer) issues
  // every TMA copy and tensor-core product, so no worker waits on a blocking MMA issue.  The two sides
  // meet at CTA-wide OR-barriers (A1, A3, A4, A5; A2 on a segment's first chunk) that also carry a
  // failed wait; the workers sync among themselves on barrier 2, and the producer tells them that a
  // context store has read wu (barrier 3, arrive / sync).
  const bool producer = warp == FWARPS;
  for (int c = cfirst; c < cend; ++c) {
    const int it = c - cfirst;
    const int stage = it & 1;
    const bool emit = outputs && c >= cbeg;  // Q, P (and the output if wanted)
    const bool emit_o = emit && want_o;
    const bool save_c = save_wy && emit;      // this chunk's context tiles
    const int t64row = ((chunk0 + c) * H + h) * T64_TILES * CH;
    const int t128row = ((chunk0 + c) * H + h) * T128_TILES * D;
    const int tok0 = bos + c * CH;
    const int nvalid = min(CH, len - c * CH);
    uint8_t *st = sm.ring[stage];
    const bool more = c + 1 < cend;
    const int nvn = more ? min(CH, len - (c + 1) * CH) : 0;
    uint8_t *stn = sm.ring[stage ^ 1];
    float *gbeta = sm.beta[stage];
    Gates &G = sm.gt[stage];

    if (producer) {
      // ================================================================ producer
      // the previous chunk's tile stores have read s0 / x1 / x2 / ah / p / its ring stage (rewritten next)
      if (lane == 0 && (save_states || save_wy)) tma_store_wait_read();
      __syncwarp();
      if (__syncthreads_or(false)) {  // A1
        failed = true;
        break;
      }
      // the next chunk into the other stage: its last reader, the previous chunk's MMA 4, completed
      if (lane == 0 && more) issue_tma(c + 1, stage ^ 1);
      if (it == 0) {
        __syncthreads_or(false);  // A2: the first chunk normalised
        if (lane == 0) {
          fence_after();
          issue_mma1(st);
        }
      }
      __syncwarp();
      if (__syncthreads_or(false)) {  // A3: Ahat, X1, X2, P and the fp16 state copy are in shared memory
        failed = true;
        break;
      }
      if (lane == 0) {
        fence_after();
        if (save_c) {  // X1, X2, Ahat and P of this (chunk, head), and its K, Q, V operand tiles
          tma_store_3d(&tmw, 0, t64row + T64_X1 * CH, 0, u32(sm.x1));
          tma_store_3d(&tmw, 0, t64row + T64_X2 * CH, 0, u32(sm.x2));
          tma_store_3d(&tmw, 0, t64row + T64_AH * CH, 0, u32(sm.ah));
          tma_store_3d(&tmw, 0, t64row + T64_P * CH, 0, u32(sm.p));
          const int qrow = ((chunk0 + c) * H + h) * TQ_TILES * CH;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            tma_store_3d(&tm3, 64 * hb, qrow + TQ_K * CH, 0, u32(st + 2 * hb * HT));
            tma_store_3d(&tm3, 64 * hb, qrow + TQ_Q * CH, 0, u32(st + (2 * hb + 1) * HT));
            tma_store_3d(&tm3, 64 * hb, qrow + TQ_V * CH, 0, u32(st + (4 + hb) * HT));
          }
        }
        if (save_states && c >= cbeg) {  // the fp16 chunk-start state, two 64-column blocks
          const int srow = ((chunk0 + c) * H + h) * D;
          tma_store_3d(&tms, 0, srow, 0, u32(sm.s0));
          tma_store_3d(&tms, 64, srow, 0, u32(sm.s0 + 2 * HT));
        }
        if (save_c || (save_states && c >= cbeg)) tma_store_commit();
        // ---- MMA 2: W^T = K^T X1^T, U^T = V^T X2^T  (M = 128, N = 64, K = 64)
        const uint32_t idesc = idesc_f16(128, 64, true, false);
        const uint32_t kb = u32(st), vb = u32(st + 4 * HT);
        const uint32_t x1b = u32(sm.x1), x2b = u32(sm.x2);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tm + TM_W, sdesc(kb + kk * 2048, 2 * HT, 1024), sdesc(x1b + kk * 32, 16, 1024), idesc, kk > 0);
        if (need_v) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(tm + TM_U, sdesc(vb + kk * 2048, HT, 1024), sdesc(x2b + kk * 32, 16, 1024), idesc, kk > 0);
        }
        mma_commit(u32(&sm.bar_mma));
        // Oi^T = S0 Q^T needs only the state copy and Q: it runs under the W^T read-out (MMA 3's commit
        // covers it)
        if (emit_o) {
          const uint32_t s0b = u32(sm.s0), qb = u32(st + HT);
          const uint32_t id_o = idesc_f16(128, 64, false, false);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
            mma_f16(tm + TM_O, sdesc(s0b + aoff, 16, 1024), sdesc(qb + aoff, 16, 1024), id_o, kk > 0);
          }
        }
      }
      __syncwarp();
      if (__syncthreads_or(false)) {  // A4: the gam-scaled W^T is in wu
        failed = true;
        break;
      }
      if (lane == 0) {
        fence_after();
        if (save_c) {  // the gam-scaled W^T tile
          tma_store_3d(&tmt, 0, t128row + T128_W * D, 0, u32(sm.wu));
          tma_store_commit();
        }
        // ---- MMA 3: Ut^T = U^T - S0 W^T   (M = 128, N = 64, K = 128)
        const uint32_t s0b = u32(sm.s0), wb = u32(sm.wu);
        const uint32_t id_u = idesc_f16(128, 64, false, true, /*neg_a=*/true);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
          mma_f16(tm + TM_U, sdesc(s0b + aoff, 16, 1024), sdesc(wb + kk * 2048, 2 * HT, 1024), id_u,
                  need_v || kk > 0);
        }
        mma_commit(u32(&sm.bar_mma));
        if (save_c) tma_store_wait_read();  // the W^T store has read wu (Ut^T is written next)
      }
      __syncwarp();
      named_bar_arrive<3, FT + 32>();
      if (__syncthreads_or(false)) {  // A5: Ut^T, Ut^T diag(cdec) and the next chunk's K, Q are ready
        failed = true;
        break;
      }
      if (lane == 0) {
        fence_after();
        if (save_c) {  // the Ut^T tile
          tma_store_3d(&tmt, 0, t128row + T128_U * D, 0, u32(sm.wu));
          tma_store_commit();
        }
        // ---- MMA 4: S += (Ut^T diag(cdec)) K (N = 128, K = 64);  Oa^T = Ut^T P^T (N = 64, K = 64)
        const uint32_t ucb = u32(sm.uc), ub = u32(sm.wu), kb = u32(st), pb = u32(sm.p);
        const uint32_t id_s = idesc_f16(128, 128, false, true);
        const uint32_t id_o = idesc_f16(128, 64, false, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tm + TM_S, sdesc(ucb + kk * 32, 16, 1024), sdesc(kb + kk * 2048, 2 * HT, 1024), id_s, true);
        if (emit_o) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(tm + TM_OA, sdesc(ub + kk * 32, 16, 1024), sdesc(pb + kk * 32, 16, 1024), id_o, kk > 0);
        }
        mma_commit(u32(&sm.bar_mma));
        if (save_c && emit_o) tma_store_wait_read();  // the Ut^T store has read wu (the O staging)
      }
      __syncwarp();
      named_bar_arrive<3, FT + 32>();
      // the next chunk's Gram product: its K, Q were normalised while MMA 3 ran; it runs during this
      // chunk's O read-out
      if (lane == 0 && more) issue_mma1(stn);
      __syncwarp();
      continue;
    }

    // ================================================================ workers
    float gnext0 = 0.f, gnext1 = 0.f;  // next chunk's log-gates (warp 0), consumed while MMA 4 runs
    if (warp == 0 && more) {
      const int tokn = bos + (c + 1) * CH;
      if (lane < nvn) gnext0 = a.g[(size_t)(tokn + lane) * H + h];
      if (lane + 32 < nvn) gnext1 = a.g[(size_t)(tokn + lane + 32) * H + h];
    }
    // g, beta of this chunk (issued one chunk ahead) must have landed before the next prefetch reuses cp.async
    cp_async_wait_all();
    if (more) issue_gb(c + 1, stage ^ 1, false);
    // chunk cfirst: wait for its tiles and normalise them here; later chunks were normalised one
    // iteration ahead, while MMA 3 and MMA 4 of the previous chunk ran
    const bool tma_ok = it > 0 || mbar_wait(u32(&sm.bar_tma[stage]), 0, err, 8);
    if (__syncthreads_or(!tma_ok || failed)) {  // A1
      failed = true;
      break;
    }
    if (it == 0) {
      if (warp == 0 && gate_prefix(sm.g[stage], G) && lane == 0 && err) atomicOr(err, 1);
      prep_kq(st, nvalid, emit, save_c ? a.nrm + ((size_t)(chunk0 + c) * H + h) * 2 * CH : nullptr);
      if (need_v) prep_v(st, nvalid);
      fence_async_smem();
      __syncthreads_or(false);  // A2: the producer issues MMA 1
    }
    {  // MMA 1: [K; Q] K^T (the first chunk here; later chunks had it issued after the previous MMA 4)
      const bool ok = mbar_wait(u32(&sm.bar_kq), kq_phase, err, 4);
      kq_phase ^= 1;
      fence_after();
      failed |= !ok;
    }

    // ---- read-out: N (fp32, rows 0-63) and P (fp16, rows 64-127); each warp takes 16 columns
    if (row < 64 || emit) {
      const int c0 = wg * 16;
      float v[16];
      tmem_ld16(tm + tm_lane + TM_KQ + c0, v);
      if (row < 64) {
        float4 *dst = reinterpret_cast<float4 *>(&sm.nf[row * LN + c0]);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        if (save_c) {  // N (fp16, row-major) straight from registers: 32 contiguous bytes per thread
          uint8_t *nt = reinterpret_cast<uint8_t *>(static_cast<f16 *>(a.t64) +
                                                    ((size_t)t64row + T64_N * CH + row) * CH + c0);
          __half2 hv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) hv[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
          reinterpret_cast<uint4 *>(nt)[0] = *reinterpret_cast<const uint4 *>(hv);
          reinterpret_cast<uint4 *>(nt)[1] = *reinterpret_cast<const uint4 *>(hv + 4);
        }
      } else {
        const int r = row - 64;
        const float gr = G.gp[r];
        float rg[16];
        ld16f(G.rgp + c0, rg);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = c0 + i <= r ? v[i] * gr * rg[i] : 0.f;
        st_chunk_f16(sm.p + chunk_off(r, c0), v);
        st_chunk_f16(sm.p + chunk_off(r, c0 + 8), v + 8);
      }
    }
    fence_before();
    fence_async_smem();  // P is an operand of MMA 4 and a context tile
    named_bar_sync<2, FT>();

    // ---- Ahat (fp32 diagonal blocks, TF32 tensor-core merges) -> X1, X2 (fp16, K-major: rows = r);
    // a saved-context forward also stages Ahat for its store (warps 0-7); meanwhile warps 8-15 copy S0
    // to its fp16 operand form and put gam_C * S0 back into TMEM (the copy is also the chunk-start state
    // that the backward reads)
    if (warp < 8) {
      wy_inverse<false, false, true>(sm.nf, LN, gbeta, sm.ys, [&](int r, int c, float a0, float a1) {
        const float2 bb = *reinterpret_cast<const float2 *>(gbeta + c), rg = *reinterpret_cast<const float2 *>(G.rgp + c);
        const float gr = G.gp[r], x0 = a0 * bb.x, x1 = a1 * bb.y;
        const uint32_t off = sw128_offset(r, c);
        *reinterpret_cast<__half2 *>(sm.x1 + off) = __floats2half2_rn(x0, x1);
        *reinterpret_cast<__half2 *>(sm.x2 + off) =
            __floats2half2_rn(c <= r ? x0 * (gr * rg.x) : 0.f, c + 1 <= r ? x1 * (gr * rg.y) : 0.f);
        if (save_wy) *reinterpret_cast<__half2 *>(sm.ah + off) = __floats2half2_rn(a0, a1);
      }, it == 0);
    } else {
      const float gC = G.gamC;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int c0 = (wg - 2) * 64 + half * 32;
        float v[32];
        tmem_ld32(tm + tm_lane + TM_S + c0, v);
        const int kb = c0 >> 6;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) st_chunk_f16(sm.s0 + kb * 2 * HT + chunk_off(row, c0 + q4 * 8), v + q4 * 8);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= gC;
        tmem_st32(tm + tm_lane + TM_S + c0, v);
      }
      fence_async_smem();  // the fp16 state copy is an operand of MMA 3 and of Oi
    }
    fence_before();
    if (__syncthreads_or(failed)) {  // A3: the producer stores the context tiles, issues MMA 2 and Oi
      failed = true;
      break;
    }
    failed |= !mma_wait();

    // ---- W^T read-out: columns scaled by gam -> fp16 MN-major B (rows = d_k)
    {
      const int c0 = wg * 16;
      float v[16];
      tmem_ld16(tm + tm_lane + TM_W + c0, v);
      float gm[16];
      ld16f(G.gam + c0, gm);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] *= gm[i];
      st_chunk_f16(sm.wu + chunk_off(row, c0), v);
      st_chunk_f16(sm.wu + chunk_off(row, c0 + 8), v + 8);
    }
    fence_before();
    fence_async_smem();
    if (__syncthreads_or(failed)) {  // A4: the producer stores W^T and issues MMA 3
      failed = true;
      break;
    }
    bool next_ok = true;
    if (more) {  // the next chunk's tiles (issued at the top of this iteration), normalised while MMA 3 runs
      next_ok = mbar_wait(u32(&sm.bar_tma[stage ^ 1]), ((it + 1) >> 1) & 1, err, 8);
      if (next_ok)
        prep_kq(stn, nvn, outputs && c + 1 >= cbeg,
                save_wy && outputs && c + 1 >= cbeg ? a.nrm + ((size_t)(chunk0 + c + 1) * H + h) * 2 * CH : nullptr);
    }
    failed |= !mma_wait();
    named_bar_sync<3, FT + 32>();  // the W^T store has read wu

    // ---- Ut^T read-out -> fp16 K-major A (rows = d_v, k = token), and Ut^T diag(cdec)
    {
      const int c0 = wg * 16;
      float v[16];
      tmem_ld16(tm + tm_lane + TM_U + c0, v);
      st_chunk_f16(sm.wu + chunk_off(row, c0), v);
      st_chunk_f16(sm.wu + chunk_off(row, c0 + 8), v + 8);
      float cd[16];
      ld16f(G.cdec + c0, cd);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] *= cd[i];
      st_chunk_f16(sm.uc + chunk_off(row, c0), v);
      st_chunk_f16(sm.uc + chunk_off(row, c0 + 8), v + 8);
    }
    fence_before();
    fence_async_smem();
    if (__syncthreads_or(failed || !next_ok)) {  // A5: the producer stores Ut^T, issues MMA 4 and the next MMA 1
      failed = true;
      break;
    }
    if (more && need_v) prep_v(stn, nvn);  // the next chunk's V, while MMA 4 runs
    fence_async_smem();
    if (warp == 0 && more) {  // gates of the next chunk, overlapping MMA 4
      float *gn = sm.g[stage ^ 1];
      gn[lane] = gnext0;
      gn[lane + 32] = gnext1;
      __syncwarp();
      if (gate_prefix(gn, sm.gt[stage ^ 1]) && lane == 0 && err) atomicOr(err, 1);
    }
    failed |= !mma_wait();
    named_bar_sync<3, FT + 32>();  // the Ut^T store has read wu

    // ---- O^T = Oi^T diag(gam) + Oa^T -> bf16 [token][d_v] staging in wu (free now) -> coalesced rows of o
    if (emit_o) {
      bf16 *stg = reinterpret_cast<bf16 *>(sm.wu);
      const int c0 = wg * 16;
      float v[16], va[16];
      tmem_ld16x2(tm + tm_lane + TM_O + c0, v, tm + tm_lane + TM_OA + c0, va);
      float gm[16];
      ld16f(G.gam + c0, gm);
#pragma unroll
      for (int i = 0; i < 16; ++i) stg[(c0 + i) * D + row] = __float2bfloat16_rn(fmaf(v[i], gm[i], va[i]));
    }
    fence_before();
    named_bar_sync<2, FT>();
    if (emit_o) {
      const uint4 *stg = reinterpret_cast<const uint4 *>(sm.wu);
      bf16 *og = static_cast<bf16 *>(a.o);
      for (int e = tid; e < CH * (D / 8); e += FT) {
        const int r = e >> 4, cc = e & 15;
        if (r < nvalid) *reinterpret_cast<uint4 *>(og + ((size_t)(tok0 + r) * H + h) * D + cc * 8) = stg[e];
      }
    }
  }

  // ---------------------------------------------------------------- end-of-segment state
  if (!failed && warp < FWARPS) {
    float *dst = nullptr;
    if (a.pass == 0) dst = (transition ? a.Mbuf : a.Ebuf) + sh_idx * DD;
    else if (j == nseg - 1 && a.ST) dst = a.ST + ((size_t)n * H + h) * DD;
    if (dst) {
      {
        const int c0 = wg * 32;
        float v[32];
        tmem_ld32(tm + tm_lane + TM_S + c0, v);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<float4 *>(dst + (size_t)row * D + c0 + 4 * q4) =
              make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
      }
    }
  }
  if (tid == FT && (save_states || save_wy)) tma_store_wait_all();
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tm, TM_COLS);
}

size_t fwd_tc_smem_bytes() { return sizeof(TcSmem) + 1024; }

int launch_fwd_tc(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                  const CUtensorMap &tw, const CUtensorMap &ts, const CUtensorMap &tt, const CUtensorMap &t3,
                  dim3 grid, cudaStream_t st) {
  const size_t smem = fwd_tc_smem_bytes();
  static_assert(sizeof(TcSmem) + 1024 <= 232448 - 256, "shared memory budget (the rest: static shared memory)");
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_pdl(fwd_tc_kernel, grid, dim3(FT + 32), smem, st, a, tq, tk, tv, tw, ts, tt, t3);
}

}  // namespace gdn
