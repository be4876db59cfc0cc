// Shared device helpers for the chunked gated delta-rule kernels (sm_103a).
//
// Tiles live in shared memory, row-major with a padded row stride.  The block
// GEMM helpers compute one warp's output tile of C = op(A) op(B) with
// mma.sync m16n8k16 (fp16 operands, fp32 accumulation) when the element type
// is fp16, and with the same fragment ownership on CUDA cores when it is fp32
// (the fp32 mode needs full fp32 products, which the bf16/tf32 tensor paths do
// not give).  The fragment layout is the PTX one for m16n8: thread `lane` owns
// rows lane/4 and lane/4 + 8, columns 2*(lane%4) + {0, 1} of every 16x8 atom.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int CH = 64;        // chunk length (tokens)
constexpr int NTHREADS = 256; // threads per CTA in the chunk kernels
constexpr int NWARPS = NTHREADS / 32;

typedef __nv_bfloat16 bf16;
typedef __half f16;

// Operand precision of the tensor-core products.  bf16 inputs are widened to
// fp16 in shared memory (exact inside fp16's range) and every computed operand
// is rounded to fp16: 11 significant bits instead of bf16's 8, at the same MMA
// rate.  Every computed operand is formed so that it stays bounded (decay
// ratios gamma_r / gamma_i <= 1 are applied before rounding).  fp32 inputs keep
// fp32 operands (CUDA-core products).
template <typename I> struct OpType;
template <> struct OpType<bf16> { typedef f16 T; };
template <> struct OpType<float> { typedef float T; };

template <typename E> struct Pad;
template <> struct Pad<bf16> { static constexpr int v = 8; };
template <> struct Pad<f16> { static constexpr int v = 8; };
template <> struct Pad<float> { static constexpr int v = 4; };

__device__ __forceinline__ float tof(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float tof(f16 x) { return __half2float(x); }
__device__ __forceinline__ float tof(float x) { return x; }
template <typename E> __device__ __forceinline__ E fromf(float x);
template <> __device__ __forceinline__ bf16 fromf<bf16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ f16 fromf<f16>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ float fromf<float>(float x) { return x; }

// store two adjacent values (columns c, c+1)
__device__ __forceinline__ void st2(bf16 *p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}
__device__ __forceinline__ void st2(f16 *p, float a, float b) {
  *reinterpret_cast<__half2 *>(p) = __floats2half2_rn(a, b);
}
__device__ __forceinline__ void st2(float *p, float a, float b) {
  *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- async copies
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
  int sz = valid ? 16 : 0;  // src-size 0 zero-fills the destination
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem), "r"(sz));
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, bool valid) {
  int sz = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// ------------------------------------------------------------------- mma.sync
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Accumulator of a warp tile WM x WN.
template <int WM, int WN> struct Acc {
  static constexpr int MI = WM / 16, NI = WN / 8;
  float c[MI][NI][4];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < MI; ++i)
#pragma unroll
      for (int j = 0; j < NI; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[i][j][e] = 0.f;
  }
  // f(row, col, float& value) for every owned element; rows/cols relative to the tile origin
  template <class F> __device__ __forceinline__ void each(F f) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < MI; ++i)
#pragma unroll
      for (int j = 0; j < NI; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) f(16 * i + (lane >> 2) + 8 * (e >> 1), 8 * j + 2 * (lane & 3) + (e & 1), c[i][j][e]);
  }
  // f(row, col, float& v0, float& v1) for each owned pair of adjacent columns
  template <class F> __device__ __forceinline__ void pairs(F f) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < MI; ++i)
#pragma unroll
      for (int j = 0; j < NI; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) f(16 * i + (lane >> 2) + 8 * h, 8 * j + 2 * (lane & 3), c[i][j][2 * h], c[i][j][2 * h + 1]);
  }
};

// One warp: acc += op(A)[m0:m0+WM, 0:K] * op(B)[0:K, n0:n0+WN].
//  AT == false: A stored [m][k] (row stride lda);  AT == true: A stored [k][m].
//  BT == false: B stored [n][k] (row stride ldb);  BT == true: B stored [k][n].
template <int WM, int WN, bool AT, bool BT>
__device__ __forceinline__ void warp_mma(Acc<WM, WN> &acc, const f16 *A, int lda, const f16 *B, int ldb, int m0,
                                         int n0, int K) {
  static_assert(WN % 16 == 0, "WN must be a multiple of 16");
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll 2
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t af[WM / 16][4];
#pragma unroll
    for (int i = 0; i < WM / 16; ++i) {
      if (!AT) {
        const f16 *p = A + (size_t)(m0 + 16 * i + (lane & 15)) * lda + k0 + (lane >> 4) * 8;
        ldsm_x4(af[i], p);
      } else {
        const f16 *p = A + (size_t)(k0 + r8 + 8 * (mi >> 1)) * lda + m0 + 16 * i + 8 * (mi & 1);
        ldsm_x4_t(af[i], p);
      }
    }
#pragma unroll
    for (int j = 0; j < WN / 16; ++j) {
      uint32_t bfr[4];
      if (!BT) {
        const f16 *p = B + (size_t)(n0 + 16 * j + r8 + 8 * (mi >> 1)) * ldb + k0 + 8 * (mi & 1);
        ldsm_x4(bfr, p);
      } else {
        const f16 *p = B + (size_t)(k0 + r8 + 8 * (mi & 1)) * ldb + n0 + 16 * j + 8 * (mi >> 1);
        ldsm_x4_t(bfr, p);
      }
#pragma unroll
      for (int i = 0; i < WM / 16; ++i) {
        mma16816(acc.c[i][2 * j], af[i], bfr[0], bfr[1]);
        mma16816(acc.c[i][2 * j + 1], af[i], bfr[2], bfr[3]);
      }
    }
  }
}

// fp32 version with identical fragment ownership, on CUDA cores.
template <int WM, int WN, bool AT, bool BT>
__device__ __forceinline__ void warp_mma(Acc<WM, WN> &acc, const float *A, int lda, const float *B, int ldb, int m0,
                                         int n0, int K) {
  const int lane = threadIdx.x & 31;
  const int r = lane >> 2, cc = 2 * (lane & 3);
#pragma unroll 2
  for (int k = 0; k < K; ++k) {
    float a[WM / 16][2], b[WN / 8][2];
#pragma unroll
    for (int i = 0; i < WM / 16; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int m = m0 + 16 * i + r + 8 * h;
        a[i][h] = AT ? A[(size_t)k * lda + m] : A[(size_t)m * lda + k];
      }
#pragma unroll
    for (int j = 0; j < WN / 8; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int n = n0 + 8 * j + cc + h;
        b[j][h] = BT ? B[(size_t)k * ldb + n] : B[(size_t)n * ldb + k];
      }
#pragma unroll
    for (int i = 0; i < WM / 16; ++i)
#pragma unroll
      for (int j = 0; j < WN / 8; ++j) {
        acc.c[i][j][0] = fmaf(a[i][0], b[j][0], acc.c[i][j][0]);
        acc.c[i][j][1] = fmaf(a[i][0], b[j][1], acc.c[i][j][1]);
        acc.c[i][j][2] = fmaf(a[i][1], b[j][0], acc.c[i][j][2]);
        acc.c[i][j][3] = fmaf(a[i][1], b[j][1], acc.c[i][j][3]);
      }
  }
}

// ------------------------------------------------------------ warp reductions
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
// sum over the 4 lanes that share an accumulator row (lane/4 equal)
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// --------------------------------------------------------------- plan tables
// Segment plan built on the device from cu_seqlens (or the uniform B x T layout).
struct Plan {
  int *seq_bos;     // [N] first token of sequence n
  int *seq_len;     // [N]
  int *seq_chunk0;  // [N] global index of the sequence's first chunk
  int *seq_seg0;    // [N] global index of the sequence's first segment
  int *seq_nseg;    // [N]
  int *seg_seq;     // [S_max] sequence of segment s, -1 if unused
  int *chunk_seq;   // [CH_max] sequence of global chunk c, -1 if unused
  int *totals;      // [2] total chunks, total segments
  int2 *chunk_info; // [CH_max] first token and valid rows of global chunk c ({0, 0} if unused)
};

constexpr float LN_EPS_WINDOW = -16.635532f;  // ln(2^-24)
constexpr int WMAX = 8;                        // longest warm-up, in chunks
constexpr float FACTOR_RANGE = 80.f;           // |G_r - G_mid| limit of the gamma factoring
constexpr float GATE_FLOOR = -128.f;           // log-gates below this decay to zero in fp32 anyway
constexpr float F16_MAX = 65504.f;             // largest finite fp16 value

// Numeric guard of the fp16 operands: true when x is not finite or would not fit fp16.  The kernels
// test the values that become operands (widened inputs, chunk-start states, dS, Ut, dUt) and set
// status bit 0 when one fails.
__device__ __forceinline__ bool f16_out(float x) { return !(fabsf(x) <= F16_MAX); }

enum StartMode { START_INIT = 0, START_WARMUP = 1, START_FIXUP = 2 };

// Segment j of a sequence covers its chunks [seg_begin(j), seg_begin(j + 1)), capped at its chunk count:
// the first segment Lfirst chunks, every later one Lseg.  A sequence of nchunks chunks has seg_count of
// them (one for an empty sequence).
__host__ __device__ __forceinline__ int seg_begin(int j, int Lfirst, int Lseg) {
  return j == 0 ? 0 : Lfirst + (j - 1) * Lseg;
}
__host__ __device__ __forceinline__ int seg_count(int nchunks, int Lfirst, int Lseg) {
  return nchunks <= Lfirst ? 1 : 1 + (nchunks - Lfirst + Lseg - 1) / Lseg;
}

// Forward: how segment (n, j) obtains its start state.  w = warm-up chunks.
__device__ __forceinline__ int fwd_start_mode(const float *gsum, int H, int h, int chunk0, int cbeg, int j,
                                              bool window, int *w) {
  *w = 0;
  if (j == 0) return START_INIT;
  if (window) {
    float acc = 0.f;
    for (int ww = 1; ww <= WMAX && ww <= cbeg; ++ww) {
      acc += gsum[(size_t)(chunk0 + cbeg - ww) * H + h];
      if (acc <= LN_EPS_WINDOW) {
        *w = ww;
        return START_WARMUP;
      }
    }
  }
  return START_FIXUP;
}

// Backward (reverse): how segment (n, j) obtains dS at its END (chunk cend).
__device__ __forceinline__ int bwd_start_mode(const float *gsum, int H, int h, int chunk0, int cend, int nchunks,
                                              int j, int nseg, bool window, int *w) {
  *w = 0;
  if (j == nseg - 1) return START_INIT;
  if (window) {
    float acc = 0.f;
    for (int ww = 1; ww <= WMAX && cend + ww <= nchunks; ++ww) {
      acc += gsum[(size_t)(chunk0 + cend + ww - 1) * H + h];
      if (acc <= LN_EPS_WINDOW) {
        *w = ww;
        return START_WARMUP;
      }
    }
  }
  return START_FIXUP;
}

// Bounded wait of one thread until *p >= target (acquire at GPU scope), polling with a short sleep;
// false when it gives up after `limit` polls (~1 s at the default).  The single-launch sequence
// parallelism waits this way for work items of other CTAs that started before it.
constexpr int PEER_WAIT_LIMIT = 1 << 22;
__device__ __forceinline__ bool wait_count_geq(const int *p, int target, int limit) {
  for (int i = 0; i < limit; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    __nanosleep(256);
  }
  return false;
}

// Programmatic dependent launch.  A kernel started with launch_pdl may be scheduled while the
// previous kernel on its stream is still finishing: it calls pdl_trigger() (its own dependents may
// then be scheduled) and pdl_wait() (returns once the previous grid has completed and its memory
// is visible) before it touches global memory.  Launched without the attribute, both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace gdn
