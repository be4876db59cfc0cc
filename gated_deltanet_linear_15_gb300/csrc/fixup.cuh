// Start-state fix-up (forward: S_start[j+1] = S_start[j] M_j + E_j over the segments of one (sequence,
// head); the reverse chain mirrors it with the segment ends), the sequential composition of the segment
// summaries (onedev.kr FlashQLA talk summary, paragraph on parallelism).  One row block (FIX_ROWS rows
// of the state) per call, run by threads 0-255 of a CTA, which synchronise on named barrier 1.  The
// composition is serial over segments, but every step's inputs (M_j and E_j's rows) are independent of
// the chain, so they stream through a two-stage shared-memory ring, two bulk copies per step issued by
// one thread on the stage's mbarrier: step i computes while step i + 1's transition lands.  The segment start modes (which segments take the fix-up at all) are
// decided up front, one segment per thread.  Used by the stand-alone fix-up kernel and, as a work item
// of the single-launch sequence parallelism, by the tcgen05 recurrent kernels.
#pragma once
#include "kernels.h"
#include "umma.cuh"

namespace gdn {

constexpr int FIX_MODES = 2048;  // segments per sequence whose modes are kept in shared memory

// shared memory of one fix-up row block: the ring, cur, the working steps, the modes, the step count and
// the ring's two mbarriers
template <int D> constexpr size_t fixup_smem_bytes() {
  return 2 * ((size_t)D * D + FIX_ROWS * D) * sizeof(float) + FIX_ROWS * D * sizeof(float) + FIX_MODES * 2 +
         FIX_MODES + 32;
}

__device__ __forceinline__ void fix_bar() { asm volatile("bar.sync 1, 256;\n" ::: "memory"); }

template <int D>
__device__ __forceinline__ void fixup_rows(const FixupArgs &a, int rb, int h, int n, unsigned char *smem) {
  using namespace umma;
  const int H = a.H;
  const int tid = threadIdx.x;
  const size_t DD = (size_t)D * D;
  float *ring = reinterpret_cast<float *>(smem);                  // 2 stages of [M (D x D) | E rows]
  float (*cur)[D] = reinterpret_cast<float (*)[D]>(ring + 2 * (DD + FIX_ROWS * D));
  short *work = reinterpret_cast<short *>(ring + 2 * (DD + FIX_ROWS * D) + FIX_ROWS * D);
  signed char *fix_mode = reinterpret_cast<signed char *>(work + FIX_MODES);
  int *nwork = reinterpret_cast<int *>(fix_mode + FIX_MODES);
  uint64_t *fbar = reinterpret_cast<uint64_t *>(fix_mode + FIX_MODES + 8);  // stage s lands on fbar[s]
  if (a.fixflag && *a.fixflag == 0) return;  // no segment of this direction needs the exact fix-up
  const int nseg = a.plan.seq_nseg[n];
  if (nseg <= 1) return;
  const int seg0 = a.plan.seq_seg0[n], chunk0 = a.plan.seq_chunk0[n];
  const int nchunks = (a.plan.seq_len[n] + CH - 1) / CH;
  const bool window = !(a.flags & kFlagWindowOff);
  constexpr int CPT = D / 32;  // columns per thread
  const int r = tid >> 5;
  const int c0 = (tid & 31) * CPT;
  const int row = rb * FIX_ROWS + r;
  // the start (end, reversed) mode of segment j
  auto start_mode = [&](int j) {
    int w;
    if (!a.reverse) return fwd_start_mode(a.gsum, H, h, chunk0, seg_begin(j, a.Lfirst, a.Lseg), j, window, &w);
    return bwd_start_mode(a.gsum, H, h, chunk0, min(seg_begin(j + 1, a.Lfirst, a.Lseg), nchunks), nchunks, j, nseg,
                          window, &w);
  };
  const bool small = nseg <= FIX_MODES;
  if (small) {
    for (int j = tid; j < nseg; j += 256) fix_mode[j] = start_mode(j) == START_FIXUP;
    fix_bar();
    if (tid == 0) {  // working steps in chain order: target jt, composed from js (forward js = jt - 1)
      int nw = 0;
      for (int step = 0; step < nseg - 1; ++step) {
        const int jt = a.reverse ? nseg - 2 - step : step + 1, js = a.reverse ? jt + 1 : jt - 1;
        if (fix_mode[jt]) work[nw++] = (short)(fix_mode[js] ? jt | 0x4000 : jt);
      }
      *nwork = nw;
    }
    fix_bar();
  }
  const int nw = small ? *nwork : nseg - 1;
  // step i -> (target jt, uses M); for very long plans the modes are evaluated on the fly
  auto step_of = [&](int i, int &jt, bool &withM) {
    if (small) {
      const int v = work[i];
      jt = v & 0x3fff;
      withM = (v & 0x4000) != 0;
      return true;
    }
    jt = a.reverse ? nseg - 2 - i : i + 1;
    if (start_mode(jt) != START_FIXUP) return false;
    withM = start_mode(a.reverse ? jt + 1 : jt - 1) == START_FIXUP;
    return true;
  };
  if (tid == 0) {
    mbar_init(smem_u32(&fbar[0]), 1);
    mbar_init(smem_u32(&fbar[1]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  fix_bar();
  // thread 0: step i's M (if used) and E rows into stage i & 1 by two bulk copies; a step with nothing to
  // load completes its stage's phase by a plain arrival
  auto issue = [&](int i) {
    if (tid != 0 || i >= nw) return;
    int jt;
    bool withM;
    const uint32_t bar = smem_u32(&fbar[i & 1]);
    if (step_of(i, jt, withM)) {
      const int js = a.reverse ? jt + 1 : jt - 1;
      const size_t src = ((size_t)(seg0 + js) * H + h) * DD;
      float *st = ring + (size_t)(i & 1) * (DD + FIX_ROWS * D);
      fence_async_smem();  // the stage's last generic reads (before the caller's barrier) precede the copies
      mbar_expect_tx(bar, (uint32_t)(((withM ? DD : 0) + FIX_ROWS * D) * sizeof(float)));
      if (withM) bulk_load(smem_u32(st), a.M + src, (uint32_t)(DD * sizeof(float)), bar);
      bulk_load(smem_u32(st + DD), a.E + src + (size_t)rb * FIX_ROWS * D, (uint32_t)(FIX_ROWS * D * sizeof(float)),
                bar);
    } else {
      mbar_arrive(bar);
    }
  };
  issue(0);
  issue(1);
  for (int i = 0; i < nw; ++i) {
    int jt;
    bool withM;
    const bool active = step_of(i, jt, withM);
    // step i's inputs have landed (step i + 1's may be in flight); an expired wait is recorded and the
    // composition goes on (its result is then not to be trusted)
    mbar_wait(smem_u32(&fbar[i & 1]), (i >> 1) & 1, a.status, 4);
    fix_bar();
    if (active) {
      const float *st = ring + (size_t)(i & 1) * (DD + FIX_ROWS * D);
      float acc[CPT];
#pragma unroll
      for (int t = 0; t < CPT; ++t) acc[t] = st[DD + r * D + c0 + t];
      if (withM) {  // cur holds the corrected state of the source segment (the previous working step)
#pragma unroll 8
        for (int k = 0; k < D; ++k) {
          const float x = cur[r][k];
          float m[CPT];
          if constexpr (CPT == 4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(st + (size_t)k * D + c0);
            m[0] = t4.x;
            m[1] = t4.y;
            m[2] = t4.z;
            m[3] = t4.w;
          } else {
            const float2 t2 = *reinterpret_cast<const float2 *>(st + (size_t)k * D + c0);
            m[0] = t2.x;
            m[1] = t2.y;
          }
#pragma unroll
          for (int t = 0; t < CPT; ++t) acc[t] = fmaf(x, m[t], acc[t]);
        }
      }
      fix_bar();  // every thread has read cur and this stage
      float *out = a.out + ((size_t)(seg0 + jt) * H + h) * DD + (size_t)row * D;
#pragma unroll
      for (int t = 0; t < CPT; ++t) {
        cur[r][c0 + t] = acc[t];
        out[c0 + t] = acc[t];
      }
    } else {
      fix_bar();
    }
    issue(i + 2);  // into the stage just read
  }
  fix_bar();  // every wait on the ring's barriers is done (every issued step was awaited)
  if (tid == 0) {
    mbar_inval(smem_u32(&fbar[0]));
    mbar_inval(smem_u32(&fbar[1]));
  }
}

}  // namespace gdn
