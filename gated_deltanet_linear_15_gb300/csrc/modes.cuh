// Fix-up modes of a call: which segment starts (forward) and ends (reverse) lie outside an effective
// sliding window and need the exact start-state fix-up (onedev.kr FlashQLA talk summary, paragraph on the
// effective sliding window: a light scan of the gate distribution decides it).  Run by one block once the
// per-(chunk, head) gate sums of the call exist: the gate scan's last block, the chunk-local half's last
// CTA (bf16, d = 128), or the plan kernel of a saved-context backward (from the forward's sums).
#pragma once
#include "kernels.h"

namespace gdn {

// Does any segment start (forward) or end (reverse) need the exact fix-up?  status[1] / status[2]
// become nonzero if so; the pass-A launches and the fix-ups of a direction without any such segment
// return at once.  With schedules (fs.hdr / bs.hdr set) it also builds each direction's work lists of
// the single-launch sequence parallelism (see Sched): pass A of segment j is needed when the start of
// segment j + 1 (forward; the end of segment j - 1 reversed) takes the fix-up, with the transition role
// too when segment j's own start (end) does.  (segment, head) pairs i0, i0 + stride, ...; gsum read
// through L2 (other blocks wrote it in this launch).  Called by one block, which synchronises itself.
static __device__ __forceinline__ bool window_ok(const float *gsum, int H, int h, int chunk0, int first, int count) {
  // the start-mode rule of the chunk kernels (fwd_start_mode / bwd_start_mode) on L2-coherent loads:
  // some w <= min(WMAX, count) with sum_{chunks first - w + 1 .. first} (forward) <= ln eps; the caller
  // passes the chunks in scan order through `first` and the direction through the sign of count
  float gs[WMAX];
  const int n = count < 0 ? -count : count;
#pragma unroll
  for (int ww = 1; ww <= WMAX; ++ww) {
    const int c = count < 0 ? first + ww - 1 : first - ww;
    gs[ww - 1] = ww <= n ? __ldcg(gsum + (size_t)(chunk0 + c) * H + h) : 0.f;
  }
  float acc = 0.f;
  bool warm = false;
#pragma unroll
  for (int ww = 1; ww <= WMAX; ++ww) {
    acc += gs[ww - 1];
    warm |= ww <= n && acc <= LN_EPS_WINDOW;
  }
  return warm;
}

static __device__ void fixup_modes(const Plan &p, const float *gsum, int H, int Lseg, int Lfirst, int S_max, unsigned flags,
                                   int *status,
                            int i0, int stride, Sched fs, Sched bs, int NH) {
  const bool window = !(flags & kFlagWindowOff);
  bool fwd_fix = false, bwd_fix = false;
  // forward start of segment j needs the fix-up (j > 0 and no certified warm-up)
  auto ffix = [&](int j, int chunk0, int h) {
    const int cbeg = seg_begin(j, Lfirst, Lseg);
    return j > 0 && !(window && window_ok(gsum, H, h, chunk0, cbeg, cbeg));
  };
  // reverse end of segment j needs the fix-up (j < nseg - 1 and no certified warm-up after it)
  auto bfix = [&](int j, int nseg, int nchunks, int chunk0, int h) {
    const int cend = min(seg_begin(j + 1, Lfirst, Lseg), nchunks);
    return j < nseg - 1 && !(window && window_ok(gsum, H, h, chunk0, cend, -(nchunks - cend)));
  };
  auto push = [](Sched &sc, int k, int v) {
    int *list = k == 0 ? sc.listA : (k == 1 ? sc.listBn : sc.listBf);
    list[atomicAdd(sc.hdr + 1 + (k == 0 ? 0 : (k == 1 ? 1 : 3)), 1)] = v;
  };
  for (int i = i0; i < S_max * H; i += stride) {
    const int s = i / H, h = i % H;
    const int n = __ldcg(p.seg_seq + s);
    if (n < 0) continue;
    const int j = s - __ldcg(p.seq_seg0 + n), nseg = __ldcg(p.seq_nseg + n), chunk0 = __ldcg(p.seq_chunk0 + n);
    const int nchunks = (__ldcg(p.seq_len + n) + CH - 1) / CH;
    const bool fj = ffix(j, chunk0, h), bj = bfix(j, nseg, nchunks, chunk0, h);
    fwd_fix |= fj;
    bwd_fix |= bj;
    const int pair = n * H + h, sh = s * H + h;
    if (fs.hdr) {
      if (j < nseg - 1 && ffix(j + 1, chunk0, h)) {
        push(fs, 0, sh * 2);
        if (fj) push(fs, 0, sh * 2 + 1);
        atomicAdd(fs.needA + pair, fj ? 2 : 1);
      }
      push(fs, fj ? 2 : 1, sh);
    }
    if (bs.hdr) {
      if (j > 0 && bfix(j - 1, nseg, nchunks, chunk0, h)) {
        push(bs, 0, sh * 2);
        if (bj) push(bs, 0, sh * 2 + 1);
        atomicAdd(bs.needA + pair, bj ? 2 : 1);
      }
      push(bs, bj ? 2 : 1, sh);
    }
  }
  if (fwd_fix) atomicOr(status + 1, 1);
  if (bwd_fix) atomicOr(status + 2, 1);
  if (!fs.hdr && !bs.hdr) return;
  __syncthreads();
  // fix-up row blocks: every (sequence, head) with a pass-A item
  for (int pair = i0; pair < NH; pair += stride) {
    if (fs.hdr && __ldcg(fs.needA + pair) > 0) fs.listF[atomicAdd(fs.hdr + 3, 1)] = pair;
    if (bs.hdr && __ldcg(bs.needA + pair) > 0) bs.listF[atomicAdd(bs.hdr + 3, 1)] = pair;
  }
}

}  // namespace gdn
