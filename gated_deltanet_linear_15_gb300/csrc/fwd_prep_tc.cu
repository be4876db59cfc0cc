// Chunk-local half of the Blackwell-native forward (bf16 inputs, d = 128): the
// (chunk, head) items are all independent; for each, it computes everything of a chunk
// that does not depend on the recurrent state and stores it as the chunk context:
//   K, Q, V operand tiles (fp16; K and Q L2-normalised, Q scaled; rows past the
//   sequence end zero) and the reciprocal norms,
//   [K; Q] K^T on the tensor cores -> N = strict_tril(K K^T), P = diag(gp) tril(Q K^T) diag(rgp),
//   Ahat = (I + diag(beta) N)^{-1} (CUDA cores, fp32, TF32 tensor-core merges),
//   X1 = Ahat diag(beta), X2 = lower(diag(gp) Ahat diag(beta rgp)).
// The recurrent kernel (fwd_tc.cu) then reads K, Q, V, X1, X2 and P by TMA and
// runs only the state-dependent products per chunk.  Splitting the chunk-local
// WY work out of the serial chain follows the four-step chunked algorithm
// (onedev.kr FlashQLA talk summary, paragraph on the WY
// representation: the intra-chunk inverse needs no state); the diagonal gamma
// scaling is pulled out of the inverse as there (paragraph on SFU load).
// Persistent CTAs, two per SM (one CTA's latency-bound phases overlap the other's),
// each loading its next item's inputs while it finishes the current one.
#include "chunk_common.cuh"
#include "kernels.h"
#include "modes.cuh"
#include "umma.cuh"

namespace gdn {

using namespace umma;

namespace {

constexpr int HT = 8192;  // one 64 x 64 fp16 half-tile, 128B-swizzled (d = 128: two per 64-row tile)
constexpr int PT = 256;   // threads per CTA (warps 0-7: the inverse's warp count)
constexpr int LN = CH + 4;

struct __align__(1024) PrepSmem {
  uint8_t kqv[6 * HT];  // [K0 | Q0 | K1 | Q1 | V0 | V1] half-tiles (0/1 = feature block)
  uint8_t x1[HT], x2[HT], ah[HT], p[HT];
  float nf[CH * LN];  // N (fp32) for the inverse, which also uses its upper triangle as scratch
  float ys[1152];
  float g[2][CH], beta[2][CH];  // per item parity: the next item's are loaded during this one
  Gates gt[2];
  uint64_t bar_tma, bar_mma;
  uint32_t tmem_base;
};

__device__ __forceinline__ uint32_t u32(const void *p) { return smem_u32(p); }

__device__ __forceinline__ void st_chunk_f16(uint8_t *dst, const float *v) {
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<uint4 *>(h);
}

}  // namespace

__global__ void __launch_bounds__(PT, 2)
    fwd_prep_tc_kernel(FwdArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmw,
                       const __grid_constant__ CUtensorMap tm3, int n_items) {
  extern __shared__ unsigned char smraw[];
  PrepSmem &sm = *reinterpret_cast<PrepSmem *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  pdl_trigger();
  pdl_wait();
  if (a.flags & kFlagDebugWaitTimeout) {  // test hook: an expiring bounded wait, then return
    __shared__ uint64_t dbg_bar;
    if (threadIdx.x == 0) debug_expire_wait(&dbg_bar, a.status, 4);
    return;
  }
  const int H = a.H;
  const bool l2 = (a.flags & kFlagL2Norm) != 0;
  // the saved-context forward and the recomputing backward keep Ahat, N and the norms too
  const bool full = a.t128 != nullptr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int *err = a.status;

  // Work items (chunk gc, head h) = (item / H, item % H), strided over the persistent CTAs (two per SM);
  // the chunks in use are the plan's first totals[0] (all of them, or none for a malformed plan).  The next
  // item's q, k, v are loaded by TMA once this item's Gram product is done and its operand tiles have left,
  // under the read-out and the inverse; its g, beta are fetched while this item's Gram product runs, from
  // its first token and valid rows, which were loaded one item earlier.
  const int tot_c = a.plan.totals[0];
  const int lim = tot_c <= n_items / H ? tot_c * H : 0;  // items of the chunks in use
  auto next_valid = [&](int item) { return item < lim ? item : n_items; };
  struct ItemInfo {
    int item, tok0, nvalid;
  };
  auto info_of = [&](int item) {
    ItemInfo r{item, 0, 0};
    if (item < n_items) {
      const int2 ci = a.plan.chunk_info[item / H];
      r.tok0 = ci.x;
      r.nvalid = ci.y;
    }
    return r;
  };
  auto issue_qkv = [&](int item, int t0) {
    const int hh = item % H;
    const uint32_t bar = u32(&sm.bar_tma);
    mbar_expect_tx(bar, 6 * HT);
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      tma_load_3d(u32(sm.kqv + 2 * hb * HT), &tmk, 64 * hb, hh, t0, bar);
      tma_load_3d(u32(sm.kqv + (2 * hb + 1) * HT), &tmq, 64 * hb, hh, t0, bar);
      tma_load_3d(u32(sm.kqv + (4 + hb) * HT), &tmv, 64 * hb, hh, t0, bar);
    }
  };
  ItemInfo cur = info_of(next_valid(blockIdx.x));
  ItemInfo nxt = info_of(next_valid(cur.item + gridDim.x));
  if (tid < 2 * CH && cur.item < n_items) {  // the first item's g, beta (later items': fetched one item ahead)
    const int r = tid & (CH - 1), hh = cur.item % H;
    const float v = r < cur.nvalid ? (tid < CH ? a.g : a.beta)[(size_t)(cur.tok0 + r) * H + hh] : 0.f;
    (tid < CH ? sm.g[0] : sm.beta[0])[r] = v;
  }
  if (tid == 0) {
    mbar_init(u32(&sm.bar_tma), 1);
    mbar_init(u32(&sm.bar_mma), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    tma_prefetch_desc(&tmw);
    tma_prefetch_desc(&tm3);
    if (cur.item < n_items) issue_qkv(cur.item, cur.tok0);
  }
  if (warp == 0) {
    tmem_alloc(u32(&sm.tmem_base), 64);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tm = sm.tmem_base;
  bool pend = cur.item < n_items;  // a q, k, v load in flight
  bool nbad = false;           // numeric guard: a widened operand out of fp16 range
  uint32_t it = 0;             // parity of both barriers: one completion each per item

  for (; cur.item < n_items; ++it) {
    const int item = cur.item, nvalid = cur.nvalid, gbuf = it & 1;
    const int t64row = item * T64_TILES * CH, qrow = item * TQ_TILES * CH;
    const bool tma_ok = mbar_wait(u32(&sm.bar_tma), it & 1, err, 8);
    pend = false;
    if (__syncthreads_or(!tma_ok)) break;

    // ---- operands: bf16 -> fp16 in place; K, Q rows L2-normalised (Q also scaled), rows >= nvalid zero.
    // For K then Q, thread t takes quarter-row t of 256: 32 features = four 16-byte chunks of one
    // 128-byte swizzled row; the four quarters of a row sit in adjacent lanes (two shuffles).
    float *nrm = full ? a.nrm + (size_t)item * 2 * CH : nullptr;
#pragma unroll 1
    for (int isq = 0; isq < 2; ++isq) {
      const int r = tid >> 2, qq = tid & 3;
      uint8_t *rowp = sm.kqv + (isq ? HT : 0) + (qq >> 1) * 2 * HT + r * 128;
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
      float rn = 1.f;
      if (l2) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float lo = __uint_as_float(raw[i] << 16), hi = __uint_as_float(raw[i] & 0xffff0000u);
          ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        rn = rsqrtf(ss + 1e-6f);
        mul *= rn;
        // normalised, every element is at most `scale` in magnitude: the fp16 range can only fail through a
        // non-finite input, which makes the squared norm non-finite (one check per row, not per element)
        nbad |= !(ss <= 3.0e38f);
      }
      if (nrm && qq == 0) nrm[(isq ? CH : 0) + r] = rn;  // 1/|k|, 1/|q| per token (1 without normalisation)
      if (r >= nvalid) mul = 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w = raw[4 * cc + i];
          const float lo = __uint_as_float(w << 16) * mul, hi = __uint_as_float(w & 0xffff0000u) * mul;
          if (!l2) nbad |= f16_out(lo) | f16_out(hi);
          const __half2 a2 = __floats2half2_rn(lo, hi);
          y[i] = *reinterpret_cast<const uint32_t *>(&a2);
        }
        *reinterpret_cast<uint4 *>(rowp + (((ch0 + cc) ^ (r & 7)) * 16)) = make_uint4(y[0], y[1], y[2], y[3]);
      }
    }
    // V: eighth-rows e of 512 (two per thread)
#pragma unroll 1
    for (int e = tid; e < 8 * CH; e += PT) {
      const int r = e >> 3, part = e & 7;
      uint8_t *rowp = sm.kqv + 4 * HT + (part >> 2) * HT + r * 128;
      const float mul = r < nvalid ? 1.f : 0.f;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int chk = (part & 3) * 2 + cc;
        uint4 q4 = *reinterpret_cast<const uint4 *>(rowp + ((chk ^ (r & 7)) * 16));
        uint32_t *w = reinterpret_cast<uint32_t *>(&q4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = __uint_as_float(w[i] << 16) * mul, hi = __uint_as_float(w[i] & 0xffff0000u) * mul;
          nbad |= f16_out(lo) | f16_out(hi);
          const __half2 a2 = __floats2half2_rn(lo, hi);
          w[i] = *reinterpret_cast<const uint32_t *>(&a2);
        }
        *reinterpret_cast<uint4 *>(rowp + ((chk ^ (r & 7)) * 16)) = q4;
      }
    }
    fence_async_smem();
    __syncthreads();

    // ---- [K; Q] K^T (M = 128, N = 64, K = 128): rows 0-63 K K^T, rows 64-127 Q K^T
    if (tid == 0) {
      fence_after();
      // the K, Q, V operand tiles are final: they leave for the context while the products run
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        tma_store_3d(&tm3, 64 * hb, qrow + TQ_K * CH, 0, u32(sm.kqv + 2 * hb * HT));
        tma_store_3d(&tm3, 64 * hb, qrow + TQ_Q * CH, 0, u32(sm.kqv + (2 * hb + 1) * HT));
        tma_store_3d(&tm3, 64 * hb, qrow + TQ_V * CH, 0, u32(sm.kqv + (4 + hb) * HT));
      }
      tma_store_commit();
      const uint32_t idesc = idesc_f16(128, 64, false, false);
      const uint32_t base = u32(sm.kqv);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (kk >> 2) * 2 * HT + (kk & 3) * 32;
        mma_f16s(tm, sdesc_s(base, 16, 1024) + (koff), sdesc_s(base, 16, 1024) + (koff), idesc, kk > 0);
      }
      mma_commit(u32(&sm.bar_mma));
      // the previous item's X1, X2, Ahat, P stores have read their staging (rewritten after the product):
      // every store group but the operand tiles just issued
      tma_store_wait_read_but_last();
    }
    __syncwarp();
    // under the Gram product: this item's gate prefix sums (warp 7; the read-out of P is their first
    // reader) and the next item's g, beta (kept in registers until the product is done)
    if (warp == PT / 32 - 1) {
      gate_prefix(sm.g[gbuf], sm.gt[gbuf]);
      if (lane == 0 && a.gsum_out) a.gsum_out[item] = sm.gt[gbuf].Glog;  // this lane wrote Glog
    }
    float gnext = 0.f;
    if (tid < 2 * CH && nxt.item < n_items) {
      const int r = tid & (CH - 1), hh = nxt.item % H;
      if (r < nxt.nvalid) gnext = (tid < CH ? a.g : a.beta)[(size_t)(nxt.tok0 + r) * H + hh];
    }
    const bool mok = mbar_wait(u32(&sm.bar_mma), it & 1, err, 4);
    fence_after();
    if (__syncthreads_or(!mok)) break;
    if (tid < 2 * CH) (tid < CH ? sm.g[gbuf ^ 1] : sm.beta[gbuf ^ 1])[tid & (CH - 1)] = gnext;
    if (tid == 0 && nxt.item < n_items) {  // kqv is free once the operand-tile stores have read it
      tma_store_wait_read();
      issue_qkv(nxt.item, nxt.tok0);
    }
    pend = nxt.item < n_items;
    // the first token and valid rows of the item after the next one, first read at the end of this item
    const int item2 = next_valid(nxt.item + gridDim.x);
    int2 ci2 = make_int2(0, 0);
    if (item2 < n_items) ci2 = a.plan.chunk_info[item2 / H];

    // ---- read-out: warp w takes TMEM lanes 32 (w % 4).. and columns 32 (w / 4)..; N (fp32, rows 0-63,
    // also stored as fp16) and P (fp16, rows 64-127)
    {
      const int row = ((warp & 3) << 5) | lane, c0 = (warp >> 2) * 32;
      float v[32];
      tmem_ld32(tm + ((uint32_t)((warp & 3) * 32) << 16) + c0, v);
      if (row < 64) {
        float4 *dst = reinterpret_cast<float4 *>(&sm.nf[row * LN + c0]);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        if (full) {  // N (fp16, row-major) straight from registers: 64 contiguous bytes per thread
          uint4 *nt = reinterpret_cast<uint4 *>(static_cast<f16 *>(a.t64) + ((size_t)t64row + T64_N * CH + row) * CH + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __half2 hv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) hv[i] = __floats2half2_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
            nt[q] = *reinterpret_cast<const uint4 *>(hv);
          }
        }
      } else {
        const int r = row - 64;
        auto pread = [&](auto pw) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float w8[8], rt[8];
            ratio8<decltype(pw)::value>(sm.gt[gbuf], r, c0 + 8 * q, rt);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int c = c0 + 8 * q + i;
              w8[i] = c <= r ? v[8 * q + i] * rt[i] : 0.f;
            }
            st_chunk_f16(sm.p + chunk_off(r, c0 + 8 * q), w8);
          }
        };
        if (sm.gt[gbuf].pw) pread(std::true_type{});
        else pread(std::false_type{});
      }
    }
    fence_before();
    __syncthreads();

    // ---- Ahat -> X1, X2 (and Ahat) staging, fp16 K-major (rows = r)
    const float *beta = sm.beta[gbuf];
    const Gates &G = sm.gt[gbuf];
    wy_inverse<false, false>(sm.nf, LN, beta, sm.ys, [&](int r, int c, float a0, float a1) {
      const float2 bb = *reinterpret_cast<const float2 *>(beta + c);
      const float x0 = a0 * bb.x, x1 = a1 * bb.y;
      const float2 rt = gratio2(G, r, c);
      const uint32_t off = sw128_offset(r, c);
      *reinterpret_cast<__half2 *>(sm.x1 + off) = __floats2half2_rn(x0, x1);
      *reinterpret_cast<__half2 *>(sm.x2 + off) =
          __floats2half2_rn(c <= r ? x0 * rt.x : 0.f, c + 1 <= r ? x1 * rt.y : 0.f);
      *reinterpret_cast<__half2 *>(sm.ah + off) = __floats2half2_rn(a0, a1);
    }, it == 0);  // ends with a proxy fence and a barrier; the zero upper blocks persist across items

    if (tid == 0) {  // X1, X2, P (and Ahat) of this (chunk, head)
      tma_store_3d(&tmw, 0, t64row + T64_X1 * CH, 0, u32(sm.x1));
      tma_store_3d(&tmw, 0, t64row + T64_X2 * CH, 0, u32(sm.x2));
      tma_store_3d(&tmw, 0, t64row + T64_P * CH, 0, u32(sm.p));
      if (full) tma_store_3d(&tmw, 0, t64row + T64_AH * CH, 0, u32(sm.ah));
      tma_store_commit();
    }
    cur = nxt;
    nxt = ItemInfo{item2, ci2.x, ci2.y};
  }
  if (nbad && err) atomicOr(err, 1);
  if (tid == 0) {
    if (pend) mbar_wait(u32(&sm.bar_tma), it & 1, err, 8);  // a load in flight lands before the CTA leaves
    tma_store_wait_all();  // the stores have read shared memory before the CTA leaves
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tm, 64);
  if (a.modes && a.gsum_out && a.status) {
    // the last CTA to finish (status[3] counts them; the plan kernel zeroed it) runs the fix-up mode scan
    // over every CTA's gate sums, which each CTA made visible before counting itself
    __shared__ int last;
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(a.status + 3, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (last) {
      __threadfence();
      Sched none;
      memset(&none, 0, sizeof none);
      fixup_modes(a.plan, a.gsum_out, H, a.Lseg, a.Lfirst, a.S_max, a.flags, a.status, tid, PT, none, none, 0);
    }
  }
}

size_t fwd_prep_tc_smem_bytes() { return sizeof(PrepSmem) + 1024; }

int launch_fwd_prep_tc(const FwdArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tw, const CUtensorMap &t3, int CH_max, cudaStream_t st) {
  if (CH_max == 0) return 0;
  const size_t smem = fwd_prep_tc_smem_bytes();
  static_assert(2 * (sizeof(PrepSmem) + 1024) <= 228 * 1024 - 2 * 1024, "two CTAs per SM");
  cudaError_t e = cudaFuncSetAttribute(fwd_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 1;
  }
  const int n_items = CH_max * a.H;
  const int grid = n_items < 2 * sms ? n_items : 2 * sms;  // persistent: two CTAs per SM
  return (int)launch_pdl(fwd_prep_tc_kernel, dim3(grid), dim3(PT), smem, st, a, tq, tk, tv, tw, t3, n_items);
}

}  // namespace gdn
