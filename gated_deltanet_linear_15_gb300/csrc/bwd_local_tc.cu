// Blackwell-native local-gradient kernel of the chunked backward (bf16 inputs,
// d = 128): persistent CTAs (one per SM, 16 warps) walk the (chunk, head) work
// items, each given the forward state S0 at the chunk start and dS at its end
// (fp16, from the two serial passes); the next item's tiles stream in by TMA
// while the current one finishes.  Every product
// is a tcgen05 MMA with fp32 accumulation in TMEM; the 64 x 64 products are
// M = 64 MMAs, whose rows spread over all four TMEM lane quarters.  The algebra is the hand-derived
// chunk backward (see bwd.cu); the WY part forms dA and dA^T as one symmetric
// matrix multiplied with K once (onedev.kr FlashQLA talk summary, paragraph on
// SFU load, last sentence).
//
// Rounds (MMA group -> read-out), TMEM regions T0..T7 of 64 columns.  The forward's chunk context
// supplies X1, X2, Ahat, P, N and Ut^T, and the reverse chain dUt^T (the operand of its own second round),
// so nothing of the forward chunk or of the chain is recomputed here.  Each round commits once the
// products its read-out needs are issued; the products read later (in brackets) are issued after that
// commit and covered by the next one, and the CUDA-core work no following product needs runs while the
// next round computes:
//   P5 dP = dO Ut^T->T0, dW'^T = -S0^T dUt^T->T1, dV^T = dUt^T X2->T6, Qa = S0^T dO^T->T5 [Kb = dS^T Ut^T->T2]
//                            under P5: <dS, S0>;  R5: dPm (over P), dP*P sums; dW'^T tile
//   P6 M1 = dW' K^T->T3, M2 = dUt V^T->T4 [Qb = K^T dPm^T->T7, Ka = Q^T dPm + dW'^T X1->T0]
//                            under P6: dv out, gam <Qa,q>;  R6: dAhat tile, beta column sums, <dV,v>
//   P7 Y1 = Ahat^T dAhat->T3 under P7: <k, Kb>, next item's gates;  R7: Y1 tile
//   P8 dT = -Y1 Ahat^T->T1   under P8: dq out;  R8: dN tile (strictly lower), beta row sums (with N)
//   P9 Ka += K^T (dN + dN^T)->T0
//                            R9: dk out (Ka + cdec Kb);  dg (reverse cumsum), dbeta
#include <cstddef>
#include <type_traits>

#include "chunk_common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {

using namespace umma;

namespace {

constexpr int D = 128;
constexpr int HT = 8192;
constexpr int LTHREADS = 512;  // 16 worker warps: four per TMEM lane quarter, 16 columns each per read-out
constexpr int LWARPS = LTHREADS / 32;
constexpr int PRODUCER = LTHREADS;       // lane 0 of warp 16 issues every product, TMA load and TMA store
constexpr int LNTHREADS = LTHREADS + 32;
constexpr uint32_t T0 = 0, T1 = 64, T2 = 128, T3 = 192, T4 = 256, T5 = 320, T6 = 384, T7 = 448;

struct __align__(1024) LocalTcSmem {
  uint8_t kq[4 * HT];   // [K0 | Q0 | K1 | Q1] half-tiles (feature blocks 0/1), rows = token
  uint8_t v[2 * HT];    // V, later Y1 (first half) and dN (second half), then the dk staging
  uint8_t dob[2 * HT];  // dO (fp16 operand form, from the chain), later the dv staging (bf16 [token][128])
  uint8_t s0[4 * HT];   // S0 [k-block][128 rows = d_v][64], later dW'^T [d_k][token]
  uint8_t ds[4 * HT];   // dS, same layout
  uint8_t p[HT];        // P, then dPm (in place)
  uint8_t x1[HT];
  uint8_t x2[HT];       // X2, later dAhat
  uint8_t ah[HT];       // Ahat (fp16); with n16, the dq staging once both are read
  uint8_t n16[HT];      // N = K K^T (fp16, [r][i], context tile)
  uint8_t wt[2 * HT];   // dUt^T [d_v][token] (the reverse chain's tile)
  uint8_t ut[2 * HT];   // Ut^T [d_v][token] (context tile)
  float g[2][CH], beta[2][CH];  // per item parity: the next item's gates are prepared during this one
  float nk[CH], nq[CH];         // reciprocal norms 1/|k|, 1/|q| (context, one bulk copy)
  Gates gt[2];
  float part[24][CH];   // per-token partial sums (reused per round)
  float acc[9][CH];     // assembled per-token terms
  float red[LWARPS];
  int nxt_info[3];       // the next item and its first token and valid rows (the producer's plan look-ups)
  uint64_t bar_a, bar_b, bar_w, bar_c, bar_mma;  // TMA: {Ut^T, dUt^T, dS, X2, S0, P, X1}, {dO}, {K, Q, norms,
                                                 // V}, {Ahat, N}; tensor cores
  uint32_t tmem_base;
};

__device__ __forceinline__ uint32_t u32(const void *p) { return smem_u32(p); }

// The r-th chunk (0 <= r < N nc) of N equal-length sequences of nc chunks, segments of F then L chunks,
// in the order of the chunk's offset within its segment, then sequence, then segment.  The reverse chain
// walks every segment at once from its last chunk to its first, so the chunks it hands over last, whose
// tiles are the likeliest to be still in L2, come first (the order changes no result: every item of the
// local kernel is independent).  Per sequence: a first segment of len0 chunks, nfull of L and a last of
// llast, so the number of segments with a chunk at offset o changes only at len0, L and llast: the
// offsets fall into at most three runs of equal width, walked here in closed form.
struct LifoOrder {
  int N, S, len0, nfull, llast, cut[3];  // cut: len0, L, llast in ascending order
};
__device__ __forceinline__ LifoOrder lifo_order(int N, int nc, int F, int L) {
  LifoOrder q;
  q.N = N;
  q.S = seg_count(nc, F, L);
  q.len0 = min(F, nc);
  q.nfull = q.S > 2 ? q.S - 2 : 0;
  q.llast = q.S > 1 ? nc - seg_begin(q.S - 1, F, L) : 0;
  int a = q.len0, b = L, c = q.llast, t;
  if (a > b) { t = a; a = b; b = t; }
  if (b > c) { t = b; b = c; c = t; }
  if (a > b) { t = a; a = b; b = t; }
  q.cut[0] = a;
  q.cut[1] = b;
  q.cut[2] = c;
  return q;
}
__device__ __forceinline__ int lifo_chunk(const LifoOrder &q, int r, int nc, int F, int L) {
  int lo = 0, base = 0;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int hi = q.cut[i];
    if (hi > lo) {
      const int m = (lo < q.len0) + (lo < L ? q.nfull : 0) + (lo < q.llast);  // segments per offset in [lo, hi)
      const int per = q.N * m, cnt = per * (hi - lo);
      if (r < base + cnt) {
        const int rr = r - base, o = lo + rr / per, idx = rr - (o - lo) * per, n = idx / m;
        int k = idx - n * m, j;
        if (o < q.len0 && k == 0) {
          j = 0;
        } else {
          k -= o < q.len0;
          j = (o < L && k < q.nfull) ? 1 + k : q.S - 1;
        }
        return n * nc + seg_begin(j, F, L) + o;
      }
      base += cnt;
      lo = hi;
    }
  }
  return r;  // not reached for r < N nc
}

__device__ __forceinline__ void st_chunk_f16(uint8_t *dst, const float *v) {
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<uint4 *>(h);
}

// 8 consecutive floats from 16-byte aligned shared memory (two vector loads, broadcast across the warp)
__device__ __forceinline__ void ld8f(const float *p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Barrier 1 over the 16 worker warps only (the producer warp does not take part), OR-reducing pred.
__device__ __forceinline__ bool wbar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n"
      ".reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.or.pred q, 1, %2, p;\n"
      "selp.u32 %0, 1, 0, q;\n"
      "}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(LTHREADS)
      : "memory");
  return r != 0;
}

// The 64-row products (dP, M1, M2, Y1, dT) are M = 64 MMAs, whose row i sits on TMEM lane 32 (i / 16) + i % 16,
// so all four lane quarters, and all 16 worker warps, share their read-outs: warp (wq, wg) reads rows 16 wq ..
// + 15, columns c0 .. c0 + 15 as one fragment (value 2m + e of lane t: row 16 wq + 8 (m & 1) + t/4, column
// c0 + 8 (m >> 1) + 2 (t%4) + e), and the row-major 64 x 64 fp16 tiles of those rows move to and from the
// same fragments by ldmatrix / stmatrix, lane t addressing row 16 wq + 8 ((t/8) & 1) + t%8 from column
// c0 + 8 ((t/8) >> 1).
__device__ __forceinline__ uint32_t rfrag_addr(const uint8_t *base, int wq, int c0, int lane) {
  const int m = lane >> 3;
  return smem_u32(base + chunk_off(16 * wq + 8 * (m & 1) + (lane & 7), c0 + 8 * (m >> 1)));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}
// sums of a row pair over the four lanes of a quad and of four columns over the eight quads of a warp
__device__ __forceinline__ void quad_sum2(float (&v)[2]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    v[h] += __shfl_xor_sync(0xffffffffu, v[h], 1);
    v[h] += __shfl_xor_sync(0xffffffffu, v[h], 2);
  }
}
__device__ __forceinline__ void col_sum4(float (&v)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[k] += __shfl_xor_sync(0xffffffffu, v[k], 4);
    v[k] += __shfl_xor_sync(0xffffffffu, v[k], 8);
    v[k] += __shfl_xor_sync(0xffffffffu, v[k], 16);
  }
}

}  // namespace

__global__ void __launch_bounds__(LNTHREADS, 1)
    bwd_local_tc_kernel(BwdArgs a, const __grid_constant__ CUtensorMap tm3, const __grid_constant__ CUtensorMap tmtc,
                        const __grid_constant__ CUtensorMap tms0, const __grid_constant__ CUtensorMap tmds,
                        const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmdq,
                        const __grid_constant__ CUtensorMap tmdk, const __grid_constant__ CUtensorMap tmdv,
                        const __grid_constant__ CUtensorMap tmu, int n_items) {
  extern __shared__ unsigned char smraw[];
  LocalTcSmem &sm =
      *reinterpret_cast<LocalTcSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  pdl_trigger();
  pdl_wait();
  if (a.flags & kFlagDebugWaitTimeout) {  // test hook: an expiring bounded wait, then return
    __shared__ uint64_t dbg_bar;
    if (threadIdx.x == 0) debug_expire_wait(&dbg_bar, a.status, 4);
    return;
  }
  const int H = a.H;
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2, wq = warp & 3;
  const int row = (wq << 5) | lane;  // TMEM lane of this thread
  const int c0 = wg * 16;            // this warp's 16 columns of a 64-column region
  const int ra = 16 * wq + (lane >> 2), ta = c0 + 2 * (lane & 3);  // rows ra, ra + 8 and columns ta, ta + 1,
                                                                    // ta + 8, ta + 9 of its M = 64 fragments
  int *err = a.status;

  if (tid == 0) {
    mbar_init(u32(&sm.bar_a), 1);
    mbar_init(u32(&sm.bar_b), 1);
    mbar_init(u32(&sm.bar_w), 1);
    mbar_init(u32(&sm.bar_c), 1);
    mbar_init(u32(&sm.bar_mma), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    for (const CUtensorMap *m : {&tm3, &tmtc, &tms0, &tmds, &tmw, &tmdq, &tmdk, &tmdv, &tmu}) tma_prefetch_desc(m);
  }
  if (warp == 0) {
    tmem_alloc(u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tm = sm.tmem_base;
  const uint32_t tl = (uint32_t)(wq * 32) << 16;
  uint32_t phase = 0;
  auto mma_done = [&]() {
    const bool r = mbar_wait(u32(&sm.bar_mma), phase, err, 4);
    phase ^= 1;
    fence_after();
    return r;
  };
  // A staged bf16 output tile (two swizzled [64 token][64 feature] halves at `stg`) to rows t0.. of head hh:
  // a full chunk by two TMA stores (the producer; the workers fenced the staging for the async proxy and
  // met it at a barrier), a partial one by coalesced 16-byte stores of the valid rows (the workers)
  auto store_tma = [&](const CUtensorMap *map, const uint8_t *stg, int hh, int t0) {
    tma_store_3d(map, 0, hh, t0, u32(stg));
    tma_store_3d(map, 64, hh, t0, u32(stg + HT));
    tma_store_commit();
  };
  auto store_rows = [&](void *gptr, const uint8_t *stg, int hh, int t0, int nv) {
    bf16 *gp = static_cast<bf16 *>(gptr);
    for (int e = tid; e < CH * (D / 8); e += LTHREADS) {
      const int r = e >> 4, cc = e & 15;
      if (r < nv)
        *reinterpret_cast<uint4 *>(gp + ((size_t)(t0 + r) * H + hh) * D + cc * 8) =
            *reinterpret_cast<const uint4 *>(stg + (cc >> 3) * HT + r * 128 + (((cc & 7) ^ (r & 7)) << 4));
    }
  };

  // Work items (chunk gc, head h): item = gc H + h; the CTAs take the ranks b, b + G, ... and rank r is
  // head r % H of chunk lifo_chunk(r / H) for equal-length sequences (the chunks the reverse chain handed
  // over last first), of chunk r / H otherwise; the chunks in use are the plan's first totals[0] (all of
  // them, or none for a malformed plan).  The tiles of the next item are loaded by TMA while this one
  // finishes.
  const int tot_c = a.plan.totals[0];
  const int lim = tot_c <= n_items / H ? tot_c * H : 0;  // ranks of the chunks in use
  auto next_valid = [&](int rank) { return rank < lim ? rank : n_items; };
  const LifoOrder lq = lifo_order(a.ord_n, a.ord_nc, a.Lfirst, a.Lseg);
  // the item, first token and valid rows of a rank (one plan look-up, done one item ahead)
  struct ItemInfo {
    int item, tok0, nvalid, rank;
  };
  auto info_of = [&](int rank) {
    ItemInfo r{n_items, 0, 0, rank};
    if (rank < n_items) {
      const int gc = a.ord_nc > 0 ? lifo_chunk(lq, rank / H, a.ord_nc, a.Lfirst, a.Lseg) : rank / H;
      const int2 ci = a.plan.chunk_info[gc];
      r.item = gc * H + rank % H;
      r.tok0 = ci.x;
      r.nvalid = ci.y;
    }
    return r;
  };
  // The tiles of an item (item = chunk * H + head) arrive in four groups, each on its own mbarrier, each
  // part issued as soon as the previous item's last reader of its buffers is done:
  //  A (bar_a, read from P5 on): Ut^T, the chain's dUt^T and dS after that item's P6 (and Kb); X2, S0, P,
  //    X1 after its P7 (which covers Ka's context part);
  //  B (bar_b): dO (fp16, from the chain), after that item's dv store;
  //  W (bar_w, read from P6 on): the K, Q operand tiles and the reciprocal norms after its dk read-out, V
  //    after its dk store (dk is staged in V's buffer);
  //  C (bar_c, read from R6 on): Ahat and N after its dq store (dq is staged in their buffers).
  // The early part of a group only raises the bytes its barrier expects; the last part arrives, so a phase
  // completes once every part has been issued and has landed.
  auto issue_a1 = [&](int item) {  // Ut^T, dUt^T, dS
    const uint32_t bar = u32(&sm.bar_a);
    const int srow = item * D;
    mbar_expect_tx_only(bar, 8 * HT);
    tma_load_3d(u32(sm.ut), &tmu, 0, (item * T128_TILES + T128_U) * D, 0, bar);
    tma_load_3d(u32(sm.wt), &tmtc, 0, (item * TC_TILES + TC_DUT) * D, 0, bar);
    tma_load_3d(u32(sm.ds), &tmds, 0, srow, 0, bar);
    tma_load_3d(u32(sm.ds + 2 * HT), &tmds, 64, srow, 0, bar);
  };
  auto issue_a2 = [&](int item) {  // X2, S0, P, X1; the group's arrival
    const uint32_t bar = u32(&sm.bar_a);
    const int row = item * T64_TILES * CH;
    mbar_expect_tx(bar, 7 * HT);
    tma_load_3d(u32(sm.x2), &tmw, 0, row + T64_X2 * CH, 0, bar);
    tma_load_3d(u32(sm.s0), &tms0, 0, item * D, 0, bar);
    tma_load_3d(u32(sm.s0 + 2 * HT), &tms0, 64, item * D, 0, bar);
    tma_load_3d(u32(sm.p), &tmw, 0, row + T64_P * CH, 0, bar);
    tma_load_3d(u32(sm.x1), &tmw, 0, row + T64_X1 * CH, 0, bar);
  };
  auto issue_c = [&](int item) {  // Ahat, N
    const uint32_t bar = u32(&sm.bar_c);
    const int row = item * T64_TILES * CH;
    mbar_expect_tx(bar, 2 * HT);
    tma_load_3d(u32(sm.ah), &tmw, 0, row + T64_AH * CH, 0, bar);
    tma_load_3d(u32(sm.n16), &tmw, 0, row + T64_N * CH, 0, bar);
  };
  auto issue_do = [&](int item) {  // dO in its fp16 operand form (the chain converted it), both feature halves
    const uint32_t bar = u32(&sm.bar_b);
    mbar_expect_tx(bar, 2 * HT);
    tma_load_3d(u32(sm.dob), &tmtc, 0, (item * TC_TILES + TC_DO) * D, 0, bar);
  };
  auto issue_w1 = [&](int item) {  // K, Q operand tiles, reciprocal norms
    const int qrow = item * TQ_TILES * CH;
    const uint32_t bar = u32(&sm.bar_w);
    mbar_expect_tx_only(bar, 4 * HT + 2 * CH * 4);
    bulk_load(u32(sm.nk), a.nrm + (size_t)item * 2 * CH, 2 * CH * 4, bar);
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      tma_load_3d(u32(sm.kq + 2 * hb * HT), &tm3, 64 * hb, qrow + TQ_K * CH, 0, bar);
      tma_load_3d(u32(sm.kq + (2 * hb + 1) * HT), &tm3, 64 * hb, qrow + TQ_Q * CH, 0, bar);
    }
  };
  auto issue_w2 = [&](int item) {  // V; the group's arrival
    const int qrow = item * TQ_TILES * CH;
    const uint32_t bar = u32(&sm.bar_w);
    mbar_expect_tx(bar, 2 * HT);
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) tma_load_3d(u32(sm.v + hb * HT), &tm3, 64 * hb, qrow + TQ_V * CH, 0, bar);
  };
  ItemInfo cur = info_of(next_valid(blockIdx.x));
  if (tid == PRODUCER && cur.item < n_items) {
    issue_a1(cur.item);
    issue_a2(cur.item);
    issue_c(cur.item);
    issue_do(cur.item);
    issue_w1(cur.item);
    issue_w2(cur.item);
  }
  // ---------------- worker warps 0-15: read-outs and the CUDA-core parts of every round
  bool failed = false, release = false;  // release: the producer still waits at a CTA-wide barrier
  uint32_t it = 0;  // parity of the TMA barriers: one completion per item
  if (warp < LWARPS) {
  for (; cur.item < n_items; ++it) {
  const int item = cur.item, h = item % H, tok0 = cur.tok0, nvalid = cur.nvalid;
  const int gbuf = it & 1;
  Gates &G = sm.gt[gbuf];
  float *const gbeta = sm.beta[gbuf];
  if (it == 0) {  // later items had g, beta and their gates prepared during the previous item
    if (tid < 64) sm.g[0][tid] = tid < nvalid ? a.g[(size_t)(tok0 + tid) * H + h] : 0.f;
    else if (tid < 128) sm.beta[0][tid - 64] = (tid - 64) < nvalid ? a.beta[(size_t)(tok0 + tid - 64) * H + h] : 0.f;
  }
  float gb_next = 0.f;  // g (tid < 64) or beta (64 <= tid < 128) of the next item, loaded under P5
  {
    const bool ok = mbar_wait(u32(&sm.bar_a), it & 1, err, 8) && mbar_wait(u32(&sm.bar_b), it & 1, err, 8);
    if (wbar_or(!ok)) {
      failed = release = true;
      break;
    }
  }
  if (it == 0 && warp == 0) gate_prefix(sm.g[0], sm.gt[0]);
  if (__syncthreads_or(false)) {  // B2: the producer issues P5
    failed = true;
    break;
  }
  // the next item, looked up by the producer before B2 (dependent global loads the workers do not wait for)
  const ItemInfo nxt{sm.nxt_info[0], sm.nxt_info[1], sm.nxt_info[2], 0};
  const int nitem = nxt.item;
  if (nitem < n_items && tid < 128) {  // the next item's g or beta, stored under P7 (its plan lookups have landed by now)
    const int r = tid & 63, nh = nitem % H;
    if (r < nxt.nvalid)
      gb_next = tid < 64 ? a.g[(size_t)(nxt.tok0 + r) * H + nh] : a.beta[(size_t)(nxt.tok0 + r) * H + nh];
  }
  {  // under P5: <dS, S0> over the whole state (both tiles share one layout, so compare byte positions)
    float acc = 0.f;
    const uint4 *A4 = reinterpret_cast<const uint4 *>(sm.s0), *B4 = reinterpret_cast<const uint4 *>(sm.ds);
#pragma unroll 2
    for (int e = tid; e < 4 * HT / 16; e += LTHREADS) {
      const uint4 x = A4[e], y = B4[e];
      const __half2 *xh = reinterpret_cast<const __half2 *>(&x), *yh = reinterpret_cast<const __half2 *>(&y);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fx = __half22float2(xh[i]), fy = __half22float2(yh[i]);
        acc += fx.x * fy.x + fx.y * fy.y;
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) sm.red[warp] = acc;
  }
  if (wbar_or(!mma_done())) {  // P5
    failed = release = true;
    break;
  }
  {
    // dP (M = 64 fragment): row and column sums of Z = dP * P; dPm = Gamma * dP (lower triangle) over P
    {
      auto r5 = [&](auto pw) {
        float v[8], rt[8];
        uint32_t pf[4], out[4];
        tmem_ld_frag1(tm + tl + T0 + c0, v);
        const uint32_t pa = rfrag_addr(sm.p, wq, c0, lane);
        ldmatrix_x4(pa, pf);
        ratio_frag<decltype(pw)::value>(G, ra, ta, rt);
        float rs[2] = {0.f, 0.f}, cs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float2 p2 = unpack_f16(pf[m]);
          float y[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int i = 2 * m + e, h = m & 1, k = 2 * (m >> 1) + e;
            const float zz = v[i] * (e ? p2.y : p2.x);
            rs[h] += zz;
            cs[k] += zz;
            y[e] = ta + 8 * (m >> 1) + e <= ra + 8 * h ? v[i] * rt[i] : 0.f;
          }
          out[m] = pack_f16(y[0], y[1]);
        }
        stmatrix_x4(pa, out);
        quad_sum2(rs);
        col_sum4(cs);
        if ((lane & 3) == 0) {  // row sums of Z, per 16-column block
          sm.part[16 + wg][ra] = rs[0];
          sm.part[16 + wg][ra + 8] = rs[1];
        }
        if (lane < 4) {  // column sums of Z, per 16-row block
          float *d = sm.part[8 + wq];
          d[ta] = cs[0]; d[ta + 1] = cs[1]; d[ta + 8] = cs[2]; d[ta + 9] = cs[3];
        }
      };
      if (G.pw) r5(std::true_type{});
      else r5(std::false_type{});
    }
    // dW'^T (lanes d_k) * gam -> s0 region (S0 is dead)
#pragma unroll 1
    for (int q4 = 0; q4 < 2; ++q4) {
      const int cb = c0 + q4 * 8;
      float v[8];
      tmem_ld8(tm + tl + T1 + cb, v);
      float gm[8];
      ld8f(G.gam + cb, gm);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] *= gm[i];
      st_chunk_f16(sm.s0 + chunk_off(row, cb), v);
    }
  }
  fence_before();
  fence_async_smem();
  {  // K, Q, V and the norms of this item (loaded at the end of the previous one)
    const bool ok = mbar_wait(u32(&sm.bar_w), it & 1, err, 8);
    if (__syncthreads_or(!ok)) {  // B4: the producer issues P6
      failed = true;
      break;
    }
  }
  if (tid < 64) {
    sm.acc[2][tid] = sm.part[16][tid] + sm.part[17][tid] + sm.part[18][tid] + sm.part[19][tid];  // row sums of dP * P
    sm.acc[3][tid] = sm.part[8][tid] + sm.part[9][tid] + sm.part[10][tid] + sm.part[11][tid];  // column sums of dP * P
  }
  {  // under P6: dV^T (lanes d_v, columns token) staged as bf16 dv[token][d_v] in dob (dO is dead; <dV, v>
     // comes with R6 as colsum(X2 M2)); gam <Qa, q^> per token over d_k (Qa = S0^T dO^T: the dO S0 part
     // of dq^ dotted with q^).  Fragment read-outs: the transposes are ldmatrix / stmatrix
    float s[4] = {0.f, 0.f, 0.f, 0.f};  // sums over this lane's features at its four tokens
#pragma unroll 1
    for (int ls = 0; ls < 32; ls += 16) {
      const uint32_t tq = tm + tl + ((uint32_t)ls << 16) + c0;
      float w[8], v[8];
      tmem_ld_frag2(tq + T6, w, tq + T5, v);
      uint32_t pk[4], qf[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) pk[m] = pack_bf16(w[2 * m], w[2 * m + 1]);
      stmatrix_x4_trans(frag_addr(sm.dob, HT, wq, ls, c0, lane), pk);
      ldmatrix_x4_trans(frag_addr(sm.kq + HT, 2 * HT, wq, ls, c0, lane), qf);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 q2 = unpack_f16(qf[m]);
        s[(m >> 1) * 2] += v[2 * m] * q2.x;
        s[(m >> 1) * 2 + 1] += v[2 * m + 1] * q2.y;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // over the eight lanes that share this lane's tokens
      s[k] += __shfl_xor_sync(0xffffffffu, s[k], 4);
      s[k] += __shfl_xor_sync(0xffffffffu, s[k], 8);
      s[k] += __shfl_xor_sync(0xffffffffu, s[k], 16);
    }
    if (lane < 4) {
      float gm[4];
      tok4(G.gam, ta, gm);
      float *dst = sm.part[20 + wq];
      dst[ta] = gm[0] * s[0];
      dst[ta + 1] = gm[1] * s[1];
      dst[ta + 8] = gm[2] * s[2];
      dst[ta + 9] = gm[3] * s[3];
    }
  }
  fence_before();
  fence_async_smem();  // the producer stores a full dv tile at B6
  if (nvalid < CH) {  // a partial one: its valid rows, once every warp has staged its part
    if (wbar_or(false)) {
      failed = release = true;
      break;
    }
    store_rows(a.dv, sm.dob, h, tok0, nvalid);
  }
  {  // P6, and Ahat and N of this item (loaded at the end of the previous one)
    const bool ok = mma_done() && mbar_wait(u32(&sm.bar_c), it & 1, err, 8);
    if (wbar_or(!ok)) {
      failed = release = true;
      break;
    }
  }
  if (tid < 64) sm.acc[5][tid] = sm.part[20][tid] + sm.part[21][tid] + sm.part[22][tid] + sm.part[23][tid];
  {
    // M1, M2 (M = 64 fragments, rows r): dAhat = beta_i (M1 + Gamma M2); beta column sums colsum_i(Ahat (M1 +
    // Gamma M2)); colsum_i(Ahat M1) (the dW'^T X1 part of dk^ dotted with k^).  Gate terms: <dW_r, W_r> =
    // rowsum_r(beta Ahat M1) and the row and column sums of X2 * M2 (X2 = Gamma Ahat diag(beta), M2 =
    // dUt V^T) over the strictly lower triangle only: a diagonal ratio gamma_r / gamma_r does not depend
    // on the gates, and leaving it out of both sums keeps the small gate gradient of a strongly decaying
    // chunk from being the difference of two large, differently rounded numbers.  X2 is read before dAhat
    // replaces it
    auto r6 = [&](auto pw) {
      float m1[8], m2[8], rt[8], bt[4];
      uint32_t af[4], xf[4], out[4];
      tmem_ld_frag2(tm + tl + T3 + c0, m1, tm + tl + T4 + c0, m2);
      const uint32_t xa = rfrag_addr(sm.x2, wq, c0, lane);
      ldmatrix_x4(rfrag_addr(sm.ah, wq, c0, lane), af);
      ldmatrix_x4(xa, xf);
      ratio_frag<decltype(pw)::value>(G, ra, ta, rt);
      tok4(gbeta, ta, bt);
      float rw[2] = {0.f, 0.f}, cs[4] = {0.f, 0.f, 0.f, 0.f}, ca[4] = {0.f, 0.f, 0.f, 0.f},
            cv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 a2 = unpack_f16(af[m]), x2 = unpack_f16(xf[m]);
        float o[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = 2 * m + e, h = m & 1, k = 2 * (m >> 1) + e;
          const int r = ra + 8 * h, col = ta + 8 * (m >> 1) + e;
          const float hv = e ? a2.y : a2.x;
          const float x = m1[i] + (col <= r ? m2[i] * rt[i] : 0.f);
          const float am = hv * m1[i];
          const float xm = col < r ? (e ? x2.y : x2.x) * m2[i] : 0.f;
          rw[h] += bt[k] * am + xm;
          cs[k] += hv * x;
          ca[k] += am;
          cv[k] += xm;
          o[e] = bt[k] * x;
        }
        out[m] = pack_f16(o[0], o[1]);
      }
      stmatrix_x4(xa, out);
      quad_sum2(rw);
      col_sum4(cs);
      col_sum4(ca);
      col_sum4(cv);
      if ((lane & 3) == 0) {  // row terms, per 16-column block
        sm.part[4 + wg][ra] = rw[0];
        sm.part[4 + wg][ra + 8] = rw[1];
      }
      if (lane < 4) {  // column terms, per 16-row block
        float *d0 = sm.part[8 + wq], *d1 = sm.part[12 + wq], *d2 = sm.part[wq];
        d0[ta] = cs[0]; d0[ta + 1] = cs[1]; d0[ta + 8] = cs[2]; d0[ta + 9] = cs[3];
        d1[ta] = ca[0]; d1[ta + 1] = ca[1]; d1[ta + 8] = ca[2]; d1[ta + 9] = ca[3];
        d2[ta] = cv[0]; d2[ta + 1] = cv[1]; d2[ta + 8] = cv[2]; d2[ta + 9] = cv[3];
      }
    };
    if (G.pw) r6(std::true_type{});
    else r6(std::false_type{});
  }
  if (tid < 128) (tid < 64 ? sm.g[gbuf ^ 1] : sm.beta[gbuf ^ 1])[tid & 63] = gb_next;  // next item's g, beta
  fence_before();
  fence_async_smem();
  if (__syncthreads_or(false)) {  // B6: the producer issues P7 and the next item's dO
    failed = true;
    break;
  }
  if (tid < 64) {
    sm.acc[6][tid] = sm.part[8][tid] + sm.part[9][tid] + sm.part[10][tid] + sm.part[11][tid];    // beta col terms
    sm.acc[7][tid] = sm.part[12][tid] + sm.part[13][tid] + sm.part[14][tid] + sm.part[15][tid];  // colsum(Ahat M1)
    sm.acc[4][tid] = sm.part[0][tid] + sm.part[1][tid] + sm.part[2][tid] + sm.part[3][tid];  // lower col sums of X2 * M2
    sm.acc[1][tid] = sm.part[4][tid] + sm.part[5][tid] + sm.part[6][tid] + sm.part[7][tid];  // <dW, W> + rows of X2 * M2
  }
  {  // under P7: <k^_t, Kb[:, t]> per token over d_k (Kb = dS^T Ut^T, so this is <Ut_t, dS k^_t>: cdec_t times it
     // is the state term y_t of the gate gradient and the cdec Kb part of k^ . dk^), Kb fragments against k^
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int ls = 0; ls < 32; ls += 16) {
      float kbv[8];
      uint32_t kf[4];
      tmem_ld_frag1(tm + tl + ((uint32_t)ls << 16) + T2 + c0, kbv);
      ldmatrix_x4_trans(frag_addr(sm.kq, 2 * HT, wq, ls, c0, lane), kf);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 k2 = unpack_f16(kf[m]);
        s4[(m >> 1) * 2] += kbv[2 * m] * k2.x;
        s4[(m >> 1) * 2 + 1] += kbv[2 * m + 1] * k2.y;
      }
    }
    col_sum4(s4);
    if (lane < 4) {
      float *d = sm.part[16 + wq];
      d[ta] = s4[0]; d[ta + 1] = s4[1]; d[ta + 8] = s4[2]; d[ta + 9] = s4[3];
    }
  }
  if (warp == 1 && nitem < n_items) gate_prefix(sm.g[gbuf ^ 1], sm.gt[gbuf ^ 1]);  // next item's gates, under P7
  if (wbar_or(!mma_done())) {  // P7
    failed = release = true;
    break;
  }
  if (tid < 64) sm.acc[0][tid] = sm.part[16][tid] + sm.part[17][tid] + sm.part[18][tid] + sm.part[19][tid];  // <k^, Kb>
  {  // R7: Y1 (M = 64 fragment) -> v (first half; V is dead)
    float v[8];
    uint32_t out[4];
    tmem_ld_frag1(tm + tl + T3 + c0, v);
#pragma unroll
    for (int m = 0; m < 4; ++m) out[m] = pack_f16(v[2 * m], v[2 * m + 1]);
    stmatrix_x4(rfrag_addr(sm.v, wq, c0, lane), out);
  }
  fence_before();
  fence_async_smem();
  if (__syncthreads_or(false)) {  // B7: the producer issues P8
    failed = true;
    break;
  }
  if (wbar_or(!mma_done())) {  // P8
    failed = release = true;
    break;
  }
  {  // R8 (M = 64 fragment of dT): dN[r][i] = beta_r dT_ri (i < r), zero elsewhere; beta row sums of dT * N
    float v[8];
    uint32_t nf[4], out[4];
    tmem_ld_frag1(tm + tl + T1 + c0, v);
    ldmatrix_x4(rfrag_addr(sm.n16, wq, c0, lane), nf);
    const float br[2] = {gbeta[ra], gbeta[ra + 8]};
    float rb[2] = {0.f, 0.f}, cn[4] = {0.f, 0.f, 0.f, 0.f};  // row sums of dT * N; column sums of dN * N
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 n2 = unpack_f16(nf[m]);
      float y[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 2 * m + e, h = m & 1, k = 2 * (m >> 1) + e;
        const bool lo = ta + 8 * (m >> 1) + e < ra + 8 * h;
        const float nv = e ? n2.y : n2.x;
        rb[h] += lo ? v[i] * nv : 0.f;
        y[e] = lo ? br[h] * v[i] : 0.f;
        cn[k] += y[e] * nv;
      }
      out[m] = pack_f16(y[0], y[1]);
    }
    stmatrix_x4(rfrag_addr(sm.v + HT, wq, c0, lane), out);
    quad_sum2(rb);
    col_sum4(cn);
    if ((lane & 3) == 0) {
      sm.part[16 + wg][ra] = rb[0];
      sm.part[16 + wg][ra + 8] = rb[1];
    }
    if (lane < 4) {
      float *d = sm.part[12 + wq];
      d[ta] = cn[0]; d[ta + 1] = cn[1]; d[ta + 8] = cn[2]; d[ta + 9] = cn[3];
    }
  }
  fence_before();
  fence_async_smem();
  if (__syncthreads_or(false)) {  // B9: the producer issues P9
    failed = true;
    break;
  }
  if (tid < 64) {  // k^ . dk^ per token: Q^T dPm, dW'^T X1, K^T (dN + dN^T) and cdec Kb parts, from sums above
    const int t = tid;
    const float rbs = sm.part[16][t] + sm.part[17][t] + sm.part[18][t] + sm.part[19][t];
    sm.acc[8][t] = sm.acc[3][t] + gbeta[t] * (sm.acc[7][t] + rbs) +
                   (sm.part[12][t] + sm.part[13][t] + sm.part[14][t] + sm.part[15][t]) + G.cdec[t] * sm.acc[0][t];
  }
  // ---- gate and beta gradients
  if (warp == LWARPS - 1) {  // under P9 (the other warps' shadow work is the k^ . dk^ sum)
    // dg_t = sum_{r >= t} dG_r + gam_C <dS, S0> + sum_{r < t} y_r: dG_r holds the terms whose decay factor
    // starts or ends at r (gamma_r of the inter-chunk output and of W; the ratios of P and X2, diagonal
    // excluded); the state terms y_r = cdec_r <Ut_r, dS k_r> (= cdec_r <k_r, Kb[:, r]>) depend on g_t only
    // for r < t (through cdec_r), so they enter by a forward exclusive scan (not as a total minus a reverse
    // partial sum)
    float dGv[2], yv[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r = lane + 32 * t;
      yv[t] = G.cdec[r] * sm.acc[0][r];
      dGv[t] = sm.acc[1][r] + sm.acc[2][r] - sm.acc[3][r] + sm.acc[5][r] - sm.acc[4][r];
    }
    float red = 0.f;
    for (int i = 0; i < LWARPS; ++i) red += sm.red[i];
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
    const float base = G.gamC * red;
    lo += base + (ylo - yv[0]);
    hi += base + (yhi - yv[1]);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r = lane + 32 * t;
      if (r < nvalid) {
        a.dg[(size_t)(tok0 + r) * H + h] = t ? hi : lo;
        a.dbeta[(size_t)(tok0 + r) * H + h] =
            sm.acc[6][r] + sm.part[16][r] + sm.part[17][r] + sm.part[18][r] + sm.part[19][r];
      }
    }
  }
  {  // under P9: dq raw = (scale dq^ - q^ (q^ . dq^) / scale) / |q|   (or scale dq^ without normalisation),
     // staged in the Ahat and N buffers (their last readers, P8 and R8, are done)
    const float rscale = 1.f / a.scale;
    float gm[4], dt[4], nqv[4];
    tok4(G.gam, ta, gm);
    if (l2) {  // q^ . dq^ = gam <Qa, q^> + sum_s dP * P (the Qb part: row sums of dP * P)
      float p1[4];
      tok4(sm.acc[5], ta, dt);
      tok4(sm.acc[2], ta, p1);
      tok4(sm.nq, ta, nqv);
#pragma unroll
      for (int k = 0; k < 4; ++k) dt[k] = (dt[k] + p1[k]) * rscale;
    }
#pragma unroll 1
    for (int ls = 0; ls < 32; ls += 16) {
      const uint32_t tq = tm + tl + ((uint32_t)ls << 16) + c0;
      float qa[8], qb[8];
      tmem_ld_frag2(tq + T5, qa, tq + T7, qb);
      uint32_t qf[4], pk[4];
      if (l2) ldmatrix_x4_trans(frag_addr(sm.kq + HT, 2 * HT, wq, ls, c0, lane), qf);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float o[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = 2 * m + e, k = (m >> 1) * 2 + e;
          const float dq = qb[i] + gm[k] * qa[i];
          if (l2) {
            const float2 q2 = unpack_f16(qf[m]);
            o[e] = (a.scale * dq - (e ? q2.y : q2.x) * dt[k]) * nqv[k];
          } else {
            o[e] = a.scale * dq;
          }
        }
        pk[m] = pack_bf16(o[0], o[1]);
      }
      stmatrix_x4_trans(frag_addr(sm.ah, HT, wq, ls, c0, lane), pk);
    }
  }
  fence_before();
  fence_async_smem();  // the producer stores a full dq tile at B10
  if (wbar_or(!mma_done())) {  // P9
    failed = release = true;
    break;
  }
  {  // R9: dk^T = Ka + cdec * Kb (lanes d_k); Jacobian; dk out
    uint8_t *const stg = sm.v;  // V's buffer (Y1 and dN are dead once P9 is done)
    float cd[4], dt[4], nkv[4];
    tok4(G.cdec, ta, cd);
    if (l2) {
      tok4(sm.acc[8], ta, dt);
      tok4(sm.nk, ta, nkv);
    }
#pragma unroll 1
    for (int ls = 0; ls < 32; ls += 16) {
      const uint32_t tq = tm + tl + ((uint32_t)ls << 16) + c0;
      float ka[8], kbv[8];
      tmem_ld_frag2(tq + T0, ka, tq + T2, kbv);
      uint32_t kf[4], pk[4];
      if (l2) ldmatrix_x4_trans(frag_addr(sm.kq, 2 * HT, wq, ls, c0, lane), kf);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float o[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = 2 * m + e, k = (m >> 1) * 2 + e;
          o[e] = ka[i] + cd[k] * kbv[i];
          if (l2) {
            const float2 k2 = unpack_f16(kf[m]);
            o[e] = (o[e] - (e ? k2.y : k2.x) * dt[k]) * nkv[k];
          }
        }
        pk[m] = pack_bf16(o[0], o[1]);
      }
      stmatrix_x4_trans(frag_addr(stg, HT, wq, ls, c0, lane), pk);
    }
  }
  fence_before();
  fence_async_smem();
  if (__syncthreads_or(false)) {  // B10: the producer stores full dq and dk tiles
    failed = true;
    break;
  }
  if (nvalid < CH) {
    store_rows(a.dq, sm.ah, h, tok0, nvalid);
    store_rows(a.dk, sm.v, h, tok0, nvalid);
    if (__syncthreads_or(false)) {  // B11: the dq and dk staging are read, the producer may load the next V, Ahat, N
      failed = true;
      break;
    }
  }
  cur = nxt;
  }
  if (release) __syncthreads_or(true);  // meet the producer at its pending CTA-wide barrier: it stops there
  } else {
  // ---------------- producer warp 16 (lane 0): every tensor-core product, TMA load and TMA store
  // Loads in flight that the workers have not waited for (pend_*), groups partly issued whose barrier still
  // lacks its arrival (open_*), and the parity of the phase each refers to.
  bool pend_a = cur.item < n_items, pend_b = pend_a, pend_w = pend_a, pend_c = pend_a, open_a = false,
       open_w = false;
  uint32_t par_a = 0, par_b = 0, par_w = 0, par_c = 0;
  // plan look-ups one item ahead: dependent global loads, done while the producer waits at B10
  ItemInfo nxt = info_of(next_valid(cur.rank + gridDim.x));
  bool deferred = false;  // this item's V, Ahat and N wait for the previous item's output stores: issued after B2
  for (; cur.item < n_items; ++it) {
    const int nitem = nxt.item;
    const bool more = nitem < n_items;
    if (lane == 0) {  // for the workers, who read it after B2
      sm.nxt_info[0] = nxt.item;
      sm.nxt_info[1] = nxt.tok0;
      sm.nxt_info[2] = nxt.nvalid;
    }
    const uint32_t npar = (it + 1) & 1;  // phase parity of the next item's loads
    const int item = cur.item, h = item % H, tok0 = cur.tok0, nvalid = cur.nvalid;
    {
      const bool f = __syncthreads_or(false);  // B2
      pend_a = pend_b = false;  // the workers waited for both (a failed wait is not repeated)
      if (f) break;
    }

    // ---- P5: dP = dO Ut^T -> T0 (M = 64); dW'^T = -S0^T dUt^T -> T1; dV^T = dUt^T X2 -> T6; Qa = S0^T dO^T -> T5
    //      (all before the commit: R5 overwrites S0 with dW'^T); then this item's V, Ahat, N once the previous item's
    //      dq and dk stores have read their staging, and Kb = dS^T Ut^T -> T2 (first read under P7: the P6 commit
    //      covers it)
    if (lane == 0) {
      fence_after();
      const uint32_t id_kmn = idesc_f16(128, 64, false, true), id_dp = idesc_f16(64, 64, false, true);
      const uint32_t id_mmn_neg = idesc_f16(128, 64, true, true, true), id_mk = idesc_f16(128, 64, true, false);
      const uint32_t dob = u32(sm.dob), ub = u32(sm.ut), sb = u32(sm.s0), dub = u32(sm.wt), x2b = u32(sm.x2);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        mma_f16s(tm + T0, sdesc_s(dob, 16, 1024) + ((kk >> 2) * HT + (kk & 3) * 32),
                 sdesc_s(ub, 2 * HT, 1024) + (kk * 2048), id_dp, kk > 0);
        mma_f16s(tm + T1, sdesc_s(sb, 2 * HT, 1024) + (kk * 2048), sdesc_s(dub, 2 * HT, 1024) + (kk * 2048), id_mmn_neg,
                 kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16s(tm + T6, sdesc_s(dub, 16, 1024) + (kk * 32), sdesc_s(x2b, HT, 1024) + (kk * 2048), id_kmn, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_f16s(tm + T5, sdesc_s(sb, 2 * HT, 1024) + (kk * 2048),
                 sdesc_s(dob, 16, 1024) + ((kk >> 2) * HT + (kk & 3) * 32), id_mk, kk > 0);
      mma_commit(u32(&sm.bar_mma));
      if (deferred) {
        tma_store_wait_read();
        issue_w2(item);
        issue_c(item);
      }
      const uint32_t id_mm = idesc_f16(128, 64, true, true), dsb = u32(sm.ds);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_f16s(tm + T2, sdesc_s(dsb, 2 * HT, 1024) + (kk * 2048), sdesc_s(ub, 2 * HT, 1024) + (kk * 2048), id_mm,
                 kk > 0);
    }
    __syncwarp();
    if (deferred) {
      open_w = false;
      pend_w = pend_c = true;
      par_c = it & 1;
      deferred = false;
    }
    {
      const bool f = __syncthreads_or(false);  // B4 (the workers waited for K, Q, V)
      pend_w = false;
      if (f) break;
    }
    // ---- P6: M1 = dW' K^T -> T3;  M2 = dUt V^T -> T4 (both M = 64);  then Qb = K^T dPm^T -> T7 and Ka's
    //      context-only part Q^T dPm + dW'^T X1 -> T0 (dP, read in R5, is dead), both first read after the P7
    //      commit, which covers them
    if (lane == 0) {
      fence_after();
      const uint32_t id_mk = idesc_f16(128, 64, true, false), id_m64 = idesc_f16(64, 64, true, false);
      const uint32_t id = idesc_f16(128, 64, true, true), id_km = idesc_f16(128, 64, false, true);
      const uint32_t kb = u32(sm.kq), pb = u32(sm.p), dwb = u32(sm.s0), dub = u32(sm.wt), vb = u32(sm.v);
      const uint32_t x1b = u32(sm.x1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t boff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
        mma_f16s(tm + T3, sdesc_s(dwb, 2 * HT, 1024) + (kk * 2048), sdesc_s(kb, 16, 1024) + (boff), id_m64, kk > 0);
        mma_f16s(tm + T4, sdesc_s(dub, 2 * HT, 1024) + (kk * 2048),
                 sdesc_s(vb, 16, 1024) + ((kk >> 2) * HT + (kk & 3) * 32), id_m64, kk > 0);
      }
      mma_commit(u32(&sm.bar_mma));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16s(tm + T7, sdesc_s(kb, 2 * HT, 1024) + (kk * 2048), sdesc_s(pb, 16, 1024) + (kk * 32), id_mk, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_f16s(tm + T0, sdesc_s(kb, 2 * HT, 1024) + (HT + kk * 2048), sdesc_s(pb, HT, 1024) + (kk * 2048), id,
                 kk > 0);
        mma_f16s(tm + T0, sdesc_s(dwb, 16, 1024) + (kk * 32), sdesc_s(x1b, HT, 1024) + (kk * 2048), id_km, true);
      }
    }
    __syncwarp();
    {
      const bool f = __syncthreads_or(false);  // B6 (the workers waited for Ahat and N)
      pend_c = false;
      if (f) break;
    }
    // ---- P7: Y1 = Ahat^T dAhat -> T3 (M = 64; M1, read in R6, is dead).  Then the dv tile (staged under P6), the
    //      next item's dO once that store has read its staging, and the next item's Ut^T, dUt^T, dS (their last
    //      readers, P5, P6 and Kb, are done)
    if (lane == 0) {
      fence_after();
      const uint32_t id_y1 = idesc_f16(64, 64, true, true);
      const uint32_t ab = u32(sm.ah), dab = u32(sm.x2);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_f16s(tm + T3, sdesc_s(ab, HT, 1024) + (kk * 2048), sdesc_s(dab, HT, 1024) + (kk * 2048), id_y1, kk > 0);
      mma_commit(u32(&sm.bar_mma));
      if (nvalid == CH) store_tma(&tmdv, sm.dob, h, tok0);
      if (more) {
        tma_store_wait_read();
        issue_do(nitem);
        issue_a1(nitem);
      }
    }
    __syncwarp();
    if (more) {
      pend_b = open_a = true;
      par_b = par_a = npar;
    }
    if (__syncthreads_or(false)) break;  // B7
    // ---- P8: dT = -Y1 Ahat^T -> T1 (M = 64); then the rest of the next item's group A: X2, S0, P, X1 (last read
    //      by Y1, P5, M1 and Ka's context part, which the P7 commit covered)
    if (lane == 0) {
      fence_after();
      const uint32_t id = idesc_f16(64, 64, false, false, true);
      const uint32_t yb = u32(sm.v), ab = u32(sm.ah);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) mma_f16s(tm + T1, sdesc_s(yb, 16, 1024) + (kk * 32),
                                              sdesc_s(ab, 16, 1024) + (kk * 32), id, kk > 0);
      mma_commit(u32(&sm.bar_mma));
      if (more) issue_a2(nitem);
    }
    __syncwarp();
    if (more) {
      open_a = false;
      pend_a = true;
    }
    if (__syncthreads_or(false)) break;  // B9
    // ---- P9: Ka += K^T (dN + dN^T) -> T0  (Ka's context-only part came with P6; Kb = dS^T Ut^T with P5, in T2)
    if (lane == 0) {
      fence_after();
      const uint32_t id_mm = idesc_f16(128, 64, true, true);
      const uint32_t id_mk = idesc_f16(128, 64, true, false);
      const uint32_t kb = u32(sm.kq), sgb = u32(sm.v + HT);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        // the dN tile read once as MN-major (dN) and once as K-major (dN^T)
        mma_f16s(tm + T0, sdesc_s(kb, 2 * HT, 1024) + (kk * 2048), sdesc_s(sgb, HT, 1024) + (kk * 2048), id_mm, true);
        mma_f16s(tm + T0, sdesc_s(kb, 2 * HT, 1024) + (kk * 2048), sdesc_s(sgb, 16, 1024) + (kk * 32), id_mk, true);
      }
      mma_commit(u32(&sm.bar_mma));
    }
    __syncwarp();
    const ItemInfo nn = info_of(next_valid(nxt.rank + gridDim.x));  // the item after the next one
    if (__syncthreads_or(false)) break;  // B10
    // dq (staged in the Ahat and N buffers) and dk (in V's buffer); the next item's K, Q and norms (R9 has read
    // them); its V, Ahat and N follow after its B2, once the stores have read the staging
    if (lane == 0) {
      if (nvalid == CH) {
        store_tma(&tmdq, sm.ah, h, tok0);
        store_tma(&tmdk, sm.v, h, tok0);
      }
      if (more) issue_w1(nitem);
    }
    __syncwarp();
    if (more) {
      open_w = true;
      par_w = npar;
    }
    if (nvalid < CH && __syncthreads_or(false)) break;  // B11
    deferred = more;
    cur = nxt;
    nxt = nn;
  }
  failed = cur.item < n_items;
  if (lane == 0) {
    if (failed) {  // let loads already in flight land before the CTA leaves (bounded waits)
      if (open_a) mbar_arrive(u32(&sm.bar_a));  // a partly issued group completes on the parts issued
      if (open_w) mbar_arrive(u32(&sm.bar_w));
      if (pend_a || open_a) mbar_wait(u32(&sm.bar_a), par_a, err, 8);
      if (pend_b) mbar_wait(u32(&sm.bar_b), par_b, err, 8);
      if (pend_w || open_w) mbar_wait(u32(&sm.bar_w), par_w, err, 8);
      if (pend_c) mbar_wait(u32(&sm.bar_c), par_c, err, 8);
    }
    tma_store_wait_all();  // output tiles written before the CTA leaves
  }
  __syncwarp();
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tm, 512);
}

static_assert(offsetof(LocalTcSmem, nk) % 16 == 0 && offsetof(LocalTcSmem, nq) == offsetof(LocalTcSmem, nk) + CH * 4,
              "the reciprocal norms arrive by one 16-byte-aligned bulk copy");

size_t bwd_local_tc_smem_bytes() { return sizeof(LocalTcSmem) + 1024; }

int launch_bwd_local_tc(const BwdArgs &a, const CUtensorMap *maps, int CH_max, cudaStream_t st) {
  if (CH_max == 0) return 0;
  const size_t smem = bwd_local_tc_smem_bytes();
  static_assert(sizeof(LocalTcSmem) + 1024 <= 232448 - 256, "shared memory budget (the rest: static shared memory)");
  cudaError_t e = cudaFuncSetAttribute(bwd_local_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 1;
  }
  const int n_items = CH_max * a.H;
  const int grid = n_items < sms ? n_items : sms;  // persistent: one CTA per SM
  return (int)launch_pdl(bwd_local_tc_kernel, dim3(grid), dim3(LNTHREADS), smem, st, a, maps[0], maps[1], maps[2],
                         maps[3], maps[4], maps[5], maps[6], maps[7], maps[8], n_items);
}

}  // namespace gdn
