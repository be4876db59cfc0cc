// Blackwell-native recurrent half of the forward (bf16 inputs, d = 128): TMA tile
// loads, tcgen05.mma with every accumulator in tensor memory (TMEM), the
// recurrent state resident in TMEM for the whole segment.  The chunk-local half
// (fwd_prep_tc.cu) has already stored each chunk's operand tiles K, Q, V (fp16,
// normalised) and its WY factors X1 = Ahat diag(beta), X2 = diag(gp) Ahat
// diag(beta rgp) and P = diag(gp) tril(Q K^T) diag(rgp); this kernel walks the
// chunks of a segment and runs only what involves the state S (onedev.kr
// FlashQLA talk summary, paragraph on the WY representation for the four steps:
// W, U from the chunk, then the state-dependent correction, output and update):
//   W^T = K^T X1^T, U^T = V^T X2^T        (MMA 2; independent of S, it runs while S is copied)
//   Ut^T = U^T - S0 W^T (negated-A MMA accumulating on U^T),   Oi^T = S0 Q^T       (MMA 3)
//   S   = gam_C S0 + (Ut^T diag(cdec)) K,  Oa^T = Ut^T P^T     (MMA 4)
//   O^T = Oi^T diag(gam) + Oa^T           (combined at read-out)
// with W^T's columns scaled by gam and a cdec-scaled copy of Ut^T made at read-out.
// Every product is an M = 128 MMA with the feature dimension on the TMEM lanes;
// operands are fp16 in 128-byte-swizzled shared memory (see umma.cuh); the state
// is kept in fp32 in TMEM and copied to fp16 once per chunk as the operand of
// MMA 3 and Oi (the copy is also the chunk-start state that the backward reads).
//
// One CTA of 16 worker warps and one producer warp per (segment, head): lane 0 of
// the producer issues every TMA copy and tensor-core product (an MMA issue blocks
// its thread while the tensor pipe's queue is full); the workers read TMEM (warp w
// reaches lanes 32 (w % 4)..; the four warps of a lane quarter split the columns)
// and do the CUDA-core work.  The tiles of chunk c+1 are loaded while chunk c runs.
#include "chunk_common.cuh"
#include "fixup.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {

using namespace umma;

namespace {

constexpr int D = 128;
constexpr int HT = 8192;  // one 64 x 64 fp16 half-tile, 128B-swizzled
constexpr int FT = 512;   // worker threads (16 warps); warp 16 is the producer
constexpr int FWARPS = FT / 32;

// TMEM columns; Oi, Oa are double-buffered by chunk parity (a chunk's o is read out during the next chunk)
constexpr uint32_t TM_S = 0, TM_W = 128, TM_U = 192, TM_O = 256, TM_OA = 320, TM_OB = 128, TM_COLS = 512;

// ring stage: [K0 | Q0 | K1 | Q1 | V0 | V1 | X1 | X2 | P] half-tiles (0/1 = feature block)
constexpr int R_K = 0, R_Q = 1, R_V = 4, R_X1 = 6, R_X2 = 7, R_P = 8, R_TILES = 9;

struct __align__(1024) TcSmem {
  uint8_t ring[2][R_TILES * HT];
  uint8_t uc[2 * HT];  // Ut^T diag(cdec) (K-major A, rows = d_v)
  uint8_t wu[2 * HT];  // W^T (MN-major B, rows = d_k), later Ut^T (K-major A, rows = d_v), then O staging
  uint8_t s0[4 * HT];  // S0 fp16 (K-major A: rows = d_v, two k-blocks of 128 rows)
  float g[2][CH];      // per ring stage
  Gates gt[2];         // per ring stage; the next chunk's gates are computed during this chunk
  uint64_t bar_tma[2];
  // tensor-core commits: MMA 3 and MMA 4 on bar_mma, MMA 2 on its own barrier (it is issued for the next
  // chunk right after MMA 4, so both could complete before the workers wait: a parity wait on one
  // barrier cannot tell two completed phases from none)
  uint64_t bar_mma, bar_mma2;
  uint32_t tmem_base;
};

__device__ __forceinline__ uint32_t u32(const void *p) { return smem_u32(p); }

// store 8 fp32 values as one 16-byte fp16 chunk
__device__ __forceinline__ void st_chunk_f16(uint8_t *dst, const float *v) {
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<uint4 *>(h);
}


}  // namespace

// One work item: segment s of head h in pass `pass` (0: pass A, role 0 the end state from zero or its
// warm-up, role 1 the transition; 1: outputs; 2: states only).  A CTA may run several items in turn: the
// first that does work allocates the TMEM columns (have_tm), which the caller frees after the last one.
__device__ __forceinline__ void fwd_tc_item(const FwdArgs &a, const CUtensorMap &tm3, const CUtensorMap &tmw,
                                            const CUtensorMap &tms, const CUtensorMap &tmt, const CUtensorMap &tmo,
                                            int s, int h, int role, int pass, bool &have_tm) {
  extern __shared__ unsigned char smraw[];
  TcSmem &sm = *reinterpret_cast<TcSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  // pass A of a call in which no segment needs the exact fix-up (status[1], set by the fix-up mode scan)
  if (pass == 0 && a.status && a.status[1] == 0) return;
  const int H = a.H;
  const int n = a.plan.seg_seq[s];
  if (n < 0) return;
  const int j = s - a.plan.seq_seg0[n], nseg = a.plan.seq_nseg[n];
  const int len = a.plan.seq_len[n], chunk0 = a.plan.seq_chunk0[n];
  const int bos = a.plan.seq_bos[n];
  const int nchunks = (len + CH - 1) / CH;
  const int cbeg = seg_begin(j, a.Lfirst, a.Lseg), cend = min(seg_begin(j + 1, a.Lfirst, a.Lseg), nchunks);
  const bool window = !(a.flags & kFlagWindowOff);
  int w = 0;
  const int mode = fwd_start_mode(a.gsum, H, h, chunk0, cbeg, j, window, &w);
  bool transition = false;
  if (pass == 0) {
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
  const bool outputs = (pass == 1);
  const bool need_v = !transition;
  // chunk-start states and the W^T, Ut^T context tiles leave shared memory by TMA stores (a pass
  // with o == NULL writes states and context but no output)
  const bool save_states = pass != 0 && a.states != nullptr;
  const bool save_wy = outputs && a.t128 != nullptr;
  const bool want_o = outputs && a.o != nullptr;
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
    mbar_init(u32(&sm.bar_mma2), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tma_prefetch_desc(&tm3);
    tma_prefetch_desc(&tmw);
    if (save_wy) tma_prefetch_desc(&tmt);
    if (save_states) tma_prefetch_desc(&tms);
    if (want_o) tma_prefetch_desc(&tmo);
  }
  if (!have_tm && warp == 0) {
    tmem_alloc(u32(&sm.tmem_base), TM_COLS);
    tmem_relinquish();
  }
  have_tm = true;
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tm = sm.tmem_base;
  const uint32_t tm_lane = (uint32_t)((warp & 3) * 32) << 16;

  // the context tiles of chunk c (K, X1; Q, P when it emits; V, X2 unless this is a transition)
  auto issue_tma = [&](int c, int stage) {
    const int item = (chunk0 + c) * H + h;
    const int qrow = item * TQ_TILES * CH, t64row = item * T64_TILES * CH;
    const bool wq = outputs && c >= cbeg;
    const uint32_t bytes = (3 + (wq ? 3 : 0) + (need_v ? 3 : 0)) * HT;
    const uint32_t bar = u32(&sm.bar_tma[stage]);
    uint8_t *st = sm.ring[stage];
    mbar_expect_tx(bar, bytes);
    tma_load_3d(u32(st + R_K * HT), &tm3, 0, qrow + TQ_K * CH, 0, bar);
    tma_load_3d(u32(st + (R_K + 2) * HT), &tm3, 64, qrow + TQ_K * CH, 0, bar);
    tma_load_3d(u32(st + R_X1 * HT), &tmw, 0, t64row + T64_X1 * CH, 0, bar);
    if (wq) {
      tma_load_3d(u32(st + R_Q * HT), &tm3, 0, qrow + TQ_Q * CH, 0, bar);
      tma_load_3d(u32(st + (R_Q + 2) * HT), &tm3, 64, qrow + TQ_Q * CH, 0, bar);
      tma_load_3d(u32(st + R_P * HT), &tmw, 0, t64row + T64_P * CH, 0, bar);
    }
    if (need_v) {
      tma_load_3d(u32(st + R_V * HT), &tm3, 0, qrow + TQ_V * CH, 0, bar);
      tma_load_3d(u32(st + (R_V + 1) * HT), &tm3, 64, qrow + TQ_V * CH, 0, bar);
      tma_load_3d(u32(st + R_X2 * HT), &tmw, 0, t64row + T64_X2 * CH, 0, bar);
    }
  };
  // MMA 2: W^T = K^T X1^T, U^T = V^T X2^T  (M = 128, N = 64, K = 64) of the chunk in ring stage `st`: needs
  // no state, so it is issued as soon as the tiles are in and the previous chunk has read TM_W, TM_U
  auto issue_mma2 = [&](const uint8_t *st) {
    const uint32_t idesc = idesc_f16(128, 64, true, false);
    const uint32_t kb = u32(st + R_K * HT), vb = u32(st + R_V * HT);
    const uint32_t x1b = u32(st + R_X1 * HT), x2b = u32(st + R_X2 * HT);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f16s(tm + TM_W, sdesc_s(kb, 2 * HT, 1024) + (kk * 2048), sdesc_s(x1b, 16, 1024) + (kk * 32), idesc, kk > 0);
    if (need_v) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16s(tm + TM_U, sdesc_s(vb, HT, 1024) + (kk * 2048), sdesc_s(x2b, 16, 1024) + (kk * 32), idesc, kk > 0);
    }
    mma_commit(u32(&sm.bar_mma2));
  };
  auto issue_g = [&](int c, int stage) {  // cp.async of the log-gates of chunk c
    const int tok0 = bos + c * CH;
    const int nvalid = min(CH, len - c * CH);
    load_scalars(sm.g[stage], a.g, H, h, tok0, nvalid, 0);
    cp_async_commit();
  };
  if (tid == FT && cfirst < cend) issue_tma(cfirst, 0);
  if (cfirst < cend) issue_g(cfirst, 0);

  // ---------------------------------------------------------------- initial state -> TMEM
  {
    const float *src = nullptr;
    if (!transition) {
      if (mode == START_INIT) src = a.S0 ? a.S0 + ((size_t)n * H + h) * DD : nullptr;
      else if (mode == START_FIXUP && pass != 0) src = a.Sstart + sh_idx * DD;
    }
    if (warp < FWARPS) {
      const int c0 = wg * 32;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int col = c0 + i;
        v[i] = src ? __ldcg(src + (size_t)row * D + col) : (transition && col == row ? 1.f : 0.f);
      }
      tmem_st32(tm + tm_lane + TM_S + c0, v);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();

  // O^T = Oi^T diag(gam) + Oa^T of a chunk (TMEM buffer at column offset obuf, its gates gt) -> bf16
  // [token][d_v] staging in uc, two swizzled [64 token][64 feature] halves: fragments (rows d_v, columns
  // token) transposed by stmatrix
  auto stage_o = [&](const Gates &gt, uint32_t obuf) {
    const int c0 = wg * 16, wq = warp & 3, ta = c0 + 2 * (lane & 3);
    float gm[4];
    tok4(gt.gam, ta, gm);
#pragma unroll 1
    for (int ls = 0; ls < 32; ls += 16) {
      const uint32_t tq = tm + tm_lane + ((uint32_t)ls << 16) + c0 + obuf;
      float v[8], va[8];
      tmem_ld_frag2(tq + TM_O, v, tq + TM_OA, va);
      uint32_t pk[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int k = (m >> 1) * 2;
        pk[m] = pack_bf16(fmaf(v[2 * m], gm[k], va[2 * m]), fmaf(v[2 * m + 1], gm[k + 1], va[2 * m + 1]));
      }
      stmatrix_x4_trans(frag_addr(sm.uc, HT, wq, ls, c0, lane), pk);
    }
  };
  int *err = a.status;
  uint32_t mma_phase = 0, mma2_phase = 0;
  bool failed = false;
  auto mma_wait = [&]() {
    const bool ok = mbar_wait(u32(&sm.bar_mma), mma_phase, err, 4);
    mma_phase ^= 1;
    fence_after();
    return ok;
  };

  // Workers and producer meet at CTA-wide OR-barriers (A1, A3, A4) that also carry a failed wait; the
  // workers sync among themselves on barrier 2, tell the producer that the previous chunk's o is staged
  // (barrier 4, arrive / sync), and the producer tells them that the W^T store has read wu (barrier 3)
  // and the o store uc (barrier 5, arrive / sync).  A chunk's o is read out under the next chunk's MMA 3, off the
  // recurrence's critical path; the segment's last one after the loop.
  const bool producer = warp == FWARPS;
  for (int c = cfirst; c < cend; ++c) {
    const int it = c - cfirst;
    const int stage = it & 1;
    const bool emit = outputs && c >= cbeg;  // Q, P (and the output if wanted)
    const bool emit_o = emit && want_o;
    const bool save_c = save_wy && emit;      // this chunk's W^T and Ut^T context tiles
    const int t128row = ((chunk0 + c) * H + h) * T128_TILES * D;
    const int tok0 = bos + c * CH;
    const int nvalid = min(CH, len - c * CH);
    uint8_t *st = sm.ring[stage];
    const bool more = c + 1 < cend;
    const int nvn = more ? min(CH, len - (c + 1) * CH) : 0;
    Gates &G = sm.gt[stage];
    const uint32_t ob = (uint32_t)stage * TM_OB;  // this chunk's Oi, Oa buffer
    // the previous chunk's o, read out under this chunk's MMA 3 (a full chunk: only a segment's last chunk
    // can be partial, and that one is read out after the loop)
    const bool prev_o = want_o && outputs && it > 0 && c - 1 >= cbeg;

    if (producer) {
      // ================================================================ producer
      // the previous chunk's stores have read s0 / wu (rewritten below)
      if (lane == 0 && (save_states || save_wy || want_o)) tma_store_wait_read();
      __syncwarp();
      if (__syncthreads_or(false)) {  // A1: this chunk's tiles have landed; the previous chunk is done
        failed = true;
        break;
      }
      if (lane == 0) {
        fence_after();
        if (it == 0) issue_mma2(st);  // later chunks: issued at the previous chunk's A4
        if (more) issue_tma(c + 1, stage ^ 1);  // its stage's last readers (the previous MMA 4) are done
      }
      __syncwarp();
      if (__syncthreads_or(false)) {  // A3: the fp16 state copy and the gam-scaled W^T are in shared memory
        failed = true;
        break;
      }
      if (lane == 0) {
        fence_after();
        if (save_c) {  // the gam-scaled W^T
          tma_store_3d(&tmt, 0, t128row + T128_W * D, 0, u32(sm.wu));
          tma_store_commit();
        }
        // ---- MMA 3: Ut^T = U^T - S0 W^T   (M = 128, N = 64, K = 128)
        const uint32_t s0b = u32(sm.s0), wb = u32(sm.wu);
        const uint32_t id_u = idesc_f16(128, 64, false, true, /*neg_a=*/true);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
          mma_f16s(tm + TM_U, sdesc_s(s0b, 16, 1024) + (aoff), sdesc_s(wb, 2 * HT, 1024) + (kk * 2048), id_u,
                   need_v || kk > 0);
        }
        mma_commit(u32(&sm.bar_mma));
        if (save_c) tma_store_wait_read();  // the W^T store has read wu (Ut^T is written next)
      }
      __syncwarp();
      named_bar_arrive<3, FT + 32>();
      named_bar_sync<4, FT + 32>();  // the workers staged the previous chunk's o in uc
      if (lane == 0 && prev_o) {  // the previous chunk's o (a full chunk) by two TMA stores
        tma_store_3d(&tmo, 0, h, tok0 - CH, u32(sm.uc));
        tma_store_3d(&tmo, 64, h, tok0 - CH, u32(sm.uc + HT));
        tma_store_commit();
        tma_store_wait_read();  // it has read uc (Ut^T diag(cdec) is written next)
      }
      __syncwarp();
      named_bar_arrive<5, FT + 32>();
      if (lane == 0) {
        if (save_states && c >= cbeg) {  // the fp16 chunk-start state, two 64-column blocks
          const int srow = ((chunk0 + c) * H + h) * D;
          tma_store_3d(&tms, 0, srow, 0, u32(sm.s0));
          tma_store_3d(&tms, 64, srow, 0, u32(sm.s0 + 2 * HT));
          tma_store_commit();
        }
        // Oi^T = S0 Q^T: read out with Oa during the next chunk (MMA 4's commit covers it)
        if (emit_o) {
          const uint32_t s0b = u32(sm.s0), qb = u32(st + R_Q * HT);
          const uint32_t id_o = idesc_f16(128, 64, false, false);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
            mma_f16s(tm + TM_O + ob, sdesc_s(s0b, 16, 1024) + (aoff), sdesc_s(qb, 16, 1024) + (aoff), id_o, kk > 0);
          }
        }
      }
      __syncwarp();
      if (__syncthreads_or(false)) {  // A4: Ut^T and Ut^T diag(cdec) are in shared memory
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
        const uint32_t ucb = u32(sm.uc), ub = u32(sm.wu), kb = u32(st + R_K * HT), pb = u32(st + R_P * HT);
        const uint32_t id_s = idesc_f16(128, 128, false, true);
        const uint32_t id_o = idesc_f16(128, 64, false, false);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16s(tm + TM_S, sdesc_s(ucb, 16, 1024) + (kk * 32), sdesc_s(kb, 2 * HT, 1024) + (kk * 2048), id_s, true);
        if (emit_o) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16s(tm + TM_OA + ob, sdesc_s(ub, 16, 1024) + (kk * 32), sdesc_s(pb, 16, 1024) + (kk * 32), id_o,
                     kk > 0);
        }
        mma_commit(u32(&sm.bar_mma));
      }
      __syncwarp();
      // MMA 2 of the next chunk once its tiles are in: TM_W and TM_U were read before A3 and A4
      if (lane == 0 && more && mbar_wait(u32(&sm.bar_tma[stage ^ 1]), ((it + 1) >> 1) & 1, err, 8)) {
        fence_after();
        issue_mma2(sm.ring[stage ^ 1]);
      }
      __syncwarp();
      continue;
    }

    // ================================================================ workers
    float gnext0 = 0.f, gnext1 = 0.f;  // next chunk's log-gates (warps 0, 1), consumed while MMA 4 runs
    if (warp < 2 && more) {
      const int tokn = bos + (c + 1) * CH;
      if (lane < nvn) gnext0 = a.g[(size_t)(tokn + lane) * H + h];
      if (lane + 32 < nvn) gnext1 = a.g[(size_t)(tokn + lane + 32) * H + h];
    }
    if (it == 0) cp_async_wait_all();  // the first chunk's gates (issued before the loop); later ones come from gnext
    const bool tma_ok = mbar_wait(u32(&sm.bar_tma[stage]), (it >> 1) & 1, err, 8);
    if (__syncthreads_or(!tma_ok || failed)) {  // A1: the producer issues MMA 2 and the next chunk's tiles
      failed = true;
      break;
    }
    if (it == 0) {  // later chunks had their gates prepared during the previous chunk
      if (warp == 0) gate_prefix(sm.g[stage], G);
      named_bar_sync<2, FT>();
    }
    // ---- S0 -> its fp16 operand form (rows = d_v), gam_C * S0 back into TMEM; warp w takes lane quarter
    // w % 4 and columns 32 (w / 4)..
    {
      const float gC = G.gamC;
      const int c0 = wg * 32;
      float v[32];
      tmem_ld32(tm + tm_lane + TM_S + c0, v);
      const int kb = c0 >> 6;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) st_chunk_f16(sm.s0 + kb * 2 * HT + chunk_off(row, c0 + q4 * 8), v + q4 * 8);
      bool bad = false;  // numeric guard: the fp16 state copy out of range
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        bad |= f16_out(v[i]);
        v[i] *= gC;
      }
      if (bad && err) atomicOr(err, 1);
      tmem_st32_issue(tm + tm_lane + TM_S + c0, v);  // completed before A4 (MMA 4 accumulates onto it)
    }
    {  // MMA 2 (its own barrier, one completion per chunk)
      failed |= !mbar_wait(u32(&sm.bar_mma2), mma2_phase, err, 4);
      mma2_phase ^= 1;
      fence_after();
    }

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
    fence_async_smem();  // the state copy and W^T are operands of MMA 3 and Oi
    if (__syncthreads_or(failed)) {  // A3: the producer stores W^T and issues MMA 3, then the state and Oi
      failed = true;
      break;
    }
    // under MMA 3: the previous chunk's o into the uc staging (uc's last reader, that chunk's MMA 4, is done)
    if (prev_o) stage_o(sm.gt[stage ^ 1], ob ^ TM_OB);
    fence_async_smem();
    named_bar_arrive<4, FT + 32>();  // the producer stores it
    failed |= !mma_wait();  // MMA 3
    named_bar_sync<3, FT + 32>();  // the W^T store has read wu

    // ---- Ut^T read-out -> fp16 K-major A (rows = d_v, k = token), and Ut^T diag(cdec)
    {
      const int c0 = wg * 16;
      float v[16];
      tmem_ld16(tm + tm_lane + TM_U + c0, v);
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 16; ++i) bad |= f16_out(v[i]);
      if (bad && err) atomicOr(err, 1);
      st_chunk_f16(sm.wu + chunk_off(row, c0), v);
      st_chunk_f16(sm.wu + chunk_off(row, c0 + 8), v + 8);
      float cd[16];
      ld16f(G.cdec + c0, cd);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] *= cd[i];
      named_bar_sync<5, FT + 32>();  // the o store has read uc
      st_chunk_f16(sm.uc + chunk_off(row, c0), v);
      st_chunk_f16(sm.uc + chunk_off(row, c0 + 8), v + 8);
    }
    tmem_wait_st();  // gam_C * S0, written back by the state copy
    fence_before();
    fence_async_smem();
    if (__syncthreads_or(failed)) {  // A4: the producer stores Ut^T and issues MMA 4
      failed = true;
      break;
    }
    if (warp < 2 && more)  // gates of the next chunk, overlapping MMA 4: a half per warp
      gate_prefix_part(gnext0, gnext1, sm.gt[stage ^ 1], 1 << warp);
    failed |= !mma_wait();  // MMA 4
  }

  tmem_wait_st();  // a loop left early may leave the state write-back in flight
  // ---------------------------------------------------------------- the last chunk's o
  {
    const int cl = cend - 1;
    const bool last_o = !failed && want_o && outputs && cl >= cbeg && cl >= cfirst;
    const int tok0 = bos + cl * CH, nvalid = min(CH, len - cl * CH);
    if (last_o && warp < FWARPS) stage_o(sm.gt[(cl - cfirst) & 1], (uint32_t)((cl - cfirst) & 1) * TM_OB);
    fence_before();
    fence_async_smem();
    __syncthreads();
    if (last_o && nvalid == CH && tid == FT) {  // a full chunk by two TMA stores
      tma_store_3d(&tmo, 0, h, tok0, u32(sm.uc));
      tma_store_3d(&tmo, 64, h, tok0, u32(sm.uc + HT));
      tma_store_commit();
    }
    if (last_o && nvalid < CH && warp < FWARPS) {  // a partial one by coalesced rows
      bf16 *og = static_cast<bf16 *>(a.o);
      for (int e = tid; e < CH * (D / 8); e += FT) {
        const int r = e >> 4, cc = e & 15;
        if (r < nvalid)
          *reinterpret_cast<uint4 *>(og + ((size_t)(tok0 + r) * H + h) * D + cc * 8) =
              *reinterpret_cast<const uint4 *>(sm.uc + (cc >> 3) * HT + r * 128 + (((cc & 7) ^ (r & 7)) << 4));
      }
    }
  }

  // ---------------------------------------------------------------- end-of-segment state
  if (!failed && warp < FWARPS) {
    float *dst = nullptr;
    if (pass == 0) dst = (transition ? a.Mbuf : a.Ebuf) + sh_idx * DD;
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
  if (tid == FT && (save_states || save_wy || want_o)) tma_store_wait_all();
  fence_before();
  __syncthreads();
  fence_after();
  if (tid == 0) {  // the next item of this CTA initialises them again
    mbar_inval(u32(&sm.bar_tma[0]));
    mbar_inval(u32(&sm.bar_tma[1]));
    mbar_inval(u32(&sm.bar_mma));
    mbar_inval(u32(&sm.bar_mma2));
  }
}

// The TMEM columns of the items a CTA ran, once all of them are done.
__device__ __forceinline__ void fwd_tc_release(bool have_tm) {
  if (!have_tm) return;
  extern __shared__ unsigned char smraw[];
  TcSmem &sm = *reinterpret_cast<TcSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  fence_before();
  __syncthreads();
  fence_after();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(sm.tmem_base, TM_COLS);
}

template <bool SCHED>
__global__ void __launch_bounds__(FT + 32, 1)
    fwd_tc_kernel(FwdArgs a, const __grid_constant__ CUtensorMap tm3, const __grid_constant__ CUtensorMap tmw,
                  const __grid_constant__ CUtensorMap tms, const __grid_constant__ CUtensorMap tmt,
                  const __grid_constant__ CUtensorMap tmo) {
  pdl_trigger();
  pdl_wait();
  int s = blockIdx.x, h = blockIdx.y, role = blockIdx.z, pass = a.pass;
  int *doneA = nullptr;  // a pass-A item reports its completion here
  bool have_tm = false;
  if (!SCHED && a.bal_pairs > 0 && pass != 0) {
    // balanced pass over equal-length sequences of bal_ns segments each (1-D grid): CTA b < bal_big runs the
    // b-th later segment (j >= 1) of the (sequence, head) pairs, every other CTA a share of the pairs' shorter
    // first segments (pairs k, k + G - bal_big, ...)
    const int ns = a.bal_ns, b = blockIdx.x, G = gridDim.x;
    if (b < a.bal_big) {
      const int pair = b / (ns - 1);
      fwd_tc_item(a, tm3, tmw, tms, tmt, tmo, (pair / a.H) * ns + 1 + b % (ns - 1), pair % a.H, 0, pass, have_tm);
    } else {
      for (int k = b - a.bal_big; k < a.bal_pairs; k += G - a.bal_big)
        fwd_tc_item(a, tm3, tmw, tms, tmt, tmo, (k / a.H) * ns, k % a.H, 0, pass, have_tm);
    }
    fwd_tc_release(have_tm);
    return;
  }
  if (!SCHED && pass == 0 && a.passA_items > 0) {
    // pass A by ticket (1-D grid of at most one CTA per SM): item t is role t & 1 of segment (t / 2) % S,
    // head (t / 2) / S (S segments); a call whose segments need no exact fix-up returns at once
    if (a.status && a.status[1] == 0) return;
    const int S = a.passA_items / (2 * a.H);  // segments
    __shared__ int tk;
    for (;;) {
      if (threadIdx.x == 0) tk = atomicAdd(a.status + 4, 1);
      __syncthreads();
      const int t = tk;
      __syncthreads();  // every thread has its ticket before thread 0 takes the next one
      if (t >= a.passA_items) break;
      fwd_tc_item(a, tm3, tmw, tms, tmt, tmo, (t >> 1) % S, (t >> 1) / S, t & 1, 0, have_tm);
    }
    fwd_tc_release(have_tm);
    return;
  }
  if (SCHED) {
    // single-launch sequence parallelism: this CTA runs the ticket-th item of the work lists (see Sched)
    __shared__ int tk, ok;
    const Sched &sc = a.sched;
    const int tid = threadIdx.x;
    if (tid == 0) tk = atomicAdd(sc.hdr, 1);
    __syncthreads();
    constexpr int NRB = D / FIX_ROWS;
    const int nA = __ldcg(sc.hdr + 1), nBn = __ldcg(sc.hdr + 2), nF = __ldcg(sc.hdr + 3), nBf = __ldcg(sc.hdr + 4);
    int t = tk;
    if (t < nA) {  // pass A
      const int e = sc.listA[t];
      s = (e >> 1) / a.H;
      h = (e >> 1) % a.H;
      role = e & 1;
      pass = 0;
      doneA = sc.doneA + a.plan.seg_seq[s] * a.H + h;
    } else if ((t -= nA) < nBn) {  // pass B from a start that needs no fix-up
      s = sc.listBn[t] / a.H;
      h = sc.listBn[t] % a.H;
      role = 0;
    } else if ((t -= nBn) < nF * NRB) {  // a fix-up row block, once its (sequence, head)'s pass A is done
      if (tid >= 256) return;
      const int pair = sc.listF[t / NRB];
      if (tid == 0) ok = wait_count_geq(sc.doneA + pair, sc.needA[pair], PEER_WAIT_LIMIT);
      fix_bar();
      if (!ok) {
        if (tid == 0 && a.status) atomicOr(a.status, 16);
        return;
      }
      __threadfence();
      FixupArgs fx;
      fx.ticket = nullptr;
      fx.plan = a.plan;
      fx.gsum = a.gsum;
      fx.E = a.Ebuf;
      fx.M = a.Mbuf;
      fx.out = a.Sstart;
      fx.H = a.H;
      fx.D = D;
      fx.Lseg = a.Lseg;
      fx.Lfirst = a.Lfirst;
      fx.flags = a.flags;
      fx.reverse = 0;
      fx.fixflag = nullptr;
      fx.status = a.status;
      extern __shared__ unsigned char smraw[];
      fixup_rows<D>(fx, t % NRB, pair % a.H, pair / a.H,
                    reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023));
      __threadfence();
      fix_bar();
      if (tid == 0) atomicAdd(sc.doneF + pair, 1);
      return;
    } else if ((t -= nF * NRB) < nBf) {  // pass B from a fixed-up start, once its fix-up blocks are done
      s = sc.listBf[t] / a.H;
      h = sc.listBf[t] % a.H;
      role = 0;
      const int pair = a.plan.seg_seq[s] * a.H + h;
      if (tid == 0) {
        const bool hook = (a.flags & kFlagDebugPeerTimeout) != 0;  // test hook: a wait that cannot succeed
        ok = wait_count_geq(sc.doneF + pair, hook ? NRB + 1 : NRB, hook ? 1024 : PEER_WAIT_LIMIT);
        if (!ok && a.status) atomicOr(a.status, 16);
      }
      __syncthreads();
      if (!ok) return;
      __threadfence();
    } else {
      return;  // a ticket past the lists: no work
    }
  }
  fwd_tc_item(a, tm3, tmw, tms, tmt, tmo, s, h, role, pass, have_tm);
  fwd_tc_release(have_tm);
  if (doneA) {  // the end state / transition stores of every thread are visible before the count
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(doneA, 1);
  }
}

size_t fwd_tc_smem_bytes() { return sizeof(TcSmem) + 1024; }

int launch_fwd_tc(const FwdArgs &a, const CUtensorMap &t3, const CUtensorMap &tw, const CUtensorMap &ts,
                  const CUtensorMap &tt, const CUtensorMap &to, dim3 grid, cudaStream_t st) {
  const size_t smem = fwd_tc_smem_bytes();
  static_assert(sizeof(TcSmem) + 1024 <= 232448 - 256, "shared memory budget (the rest: static shared memory)");
  static_assert(fixup_smem_bytes<D>() <= sizeof(TcSmem), "a fix-up row block fits the kernel's shared memory");
  auto kern = a.sched_on ? fwd_tc_kernel<true> : fwd_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  return (int)launch_pdl(kern, grid, dim3(FT + 32), smem, st, a, t3, tw, ts, tt, to);
}

}  // namespace gdn
