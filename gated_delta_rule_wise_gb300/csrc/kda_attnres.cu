// kda_attnres.cu -- AttnRes depth mixing ("22,580: From GPT-2 to Kimi K3"
// (yichencityu.github.io), section 12, block_attn_res): for each token row,
// the N+1 stacked block representations V_n are RMS-normalised into keys,
// scored by a learned vector w, weighted by a softmax over the block axis and
// summed:  h = sum_n softmax_n(w . V_n / rms(V_n)) V_n.
//
// HBM-bound (about N+2 row reads and one row write per token).  One CTA of
// 256 threads per row (grid-stride over rows).  Pass 1: every thread reads
// its 16-byte pieces of all blocks at once (a kernel per block count up to
// 16; above that, eight blocks at a time under a predicate) and accumulates
// w . V_n and V_n . V_n; a block reduction and one warp's softmax give the
// weights.  Pass 2 reads the same pieces again (from L2: the row was just
// read) and writes the weighted sum; both as streaming accesses, so that they
// do not evict rows that other CTAs have read once and will read again.  The
// fixed-count kernel prefetches the first two blocks of its next row into L2
// during pass 2.
#include <utility>

#include "kda_launch.cuh"

namespace kda {
namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kMaxBlocks = 32;
constexpr int kGroup = 8;  // blocks whose loads are in flight together (general kernel)
constexpr int kFixedMax = 16;  // block counts with a kernel of their own

// A row is read twice.  The first read caches it in L2 only (`first`); the
// second is its last use and reads it as streaming (`last`: evict-first), and
// the output row is stored as streaming too, so neither pushes rows that are
// still between their two reads out of L2.
enum class Use { first, last };
__device__ __forceinline__ uint4 ld16(const void *p, Use u) {
  const uint4 *q = reinterpret_cast<const uint4 *>(p);
  return u == Use::first ? __ldcg(q) : __ldcs(q);
}

template <typename T>
struct Piece;  // 16 bytes of a row
template <>
struct Piece<float> {
  static constexpr int E = 4;
  __device__ static void load(const float *p, float *x, Use use) {
    const uint4 u = ld16(p, use);
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
  }
  __device__ static void store(float *p, const float *x) {
    __stcs(reinterpret_cast<float4 *>(p), make_float4(x[0], x[1], x[2], x[3]));
  }
};
template <>
struct Piece<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ static void load(const __nv_bfloat16 *p, float *x, Use use) {
    const uint4 u = ld16(p, use);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
      x[2 * i] = __low2float(h);
      x[2 * i + 1] = __high2float(h);
    }
  }
  __device__ static void store(__nv_bfloat16 *p, const float *x) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    __stcs(reinterpret_cast<uint4 *>(p), make_uint4(w[0], w[1], w[2], w[3]));
  }
};

template <typename T>
__global__ void __launch_bounds__(kAttnThreads)
attn_res_kernel(const T *__restrict__ V, int nb, const float *__restrict__ w, T *__restrict__ h,
                long long rows, int D, float eps) {
  using P = Piece<T>;
  constexpr int E = P::E;
  __shared__ float red[kAttnWarps][kMaxBlocks][2];
  __shared__ float alpha[kMaxBlocks];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npieces = D / E;
  const size_t stride = (size_t)rows * D;  // between blocks

  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const T *vr = V + (size_t)row * D;
    // pass 1, eight blocks at a time: w . V_n and V_n . V_n
    for (int g = 0; g < nb; g += kGroup) {
      float dot[kGroup], ss[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j) dot[j] = ss[j] = 0.f;
      for (int pc = tid; pc < npieces; pc += kAttnThreads) {
        float wv[E];
        {
          const float4 *wp = reinterpret_cast<const float4 *>(w + (size_t)pc * E);
#pragma unroll
          for (int i = 0; i < E / 4; ++i) {
            const float4 u = __ldg(wp + i);
            wv[4 * i] = u.x; wv[4 * i + 1] = u.y; wv[4 * i + 2] = u.z; wv[4 * i + 3] = u.w;
          }
        }
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          if (g + j < nb) {
            float x[E];
            P::load(vr + (size_t)(g + j) * stride + (size_t)pc * E, x, Use::first);
#pragma unroll
            for (int e = 0; e < E; ++e) {
              dot[j] += wv[e] * x[e];
              ss[j] += x[e] * x[e];
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        float a = dot[j], b = ss[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          a += __shfl_xor_sync(0xffffffffu, a, off);
          b += __shfl_xor_sync(0xffffffffu, b, off);
        }
        if (lane == 0 && g + j < nb) {
          red[warp][g + j][0] = a;
          red[warp][g + j][1] = b;
        }
      }
    }
    __syncthreads();
    if (warp == 0) {  // lane n: the logit of block n, then the softmax over lanes
      float logit = -INFINITY;
      if (lane < nb) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int i = 0; i < kAttnWarps; ++i) {
          a += red[i][lane][0];
          b += red[i][lane][1];
        }
        logit = a * rsqrtf(b / (float)D + eps);
      }
      float m = logit;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      const float e = lane < nb ? __expf(logit - m) : 0.f;
      float sum = e;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane < nb) alpha[lane] = e / sum;
    }
    __syncthreads();
    // pass 2: h = sum_n alpha_n V_n, the pieces read again (from L2)
    T *hr = h + (size_t)row * D;
    for (int pc = tid; pc < npieces; pc += kAttnThreads) {
      float acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.f;
      for (int g = 0; g < nb; g += kGroup) {
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          if (g + j < nb) {
            float x[E];
            P::load(vr + (size_t)(g + j) * stride + (size_t)pc * E, x, Use::last);
            const float an = alpha[g + j];
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] += an * x[e];
          }
        }
      }
      P::store(hr + (size_t)pc * E, acc);
    }
    __syncthreads();  // red / alpha reused by the next row
  }
}

// The same with the block count fixed at compile time (1..16): every piece's
// loads for all blocks are issued together and the sums live in registers.
// Four CTAs per SM where a thread's pieces fit in 64 registers (bf16 up to
// 11 blocks, float32 up to 7), three otherwise: more rows in flight per SM
// hide more of each row's reduction than deeper unrolling within a row does.
template <typename T, int NB>
constexpr int attn_min_blocks() {
  return (sizeof(T) == 2 ? NB <= 11 : NB <= 7) ? 4 : 3;
}
template <typename T, int NB>
__global__ void __launch_bounds__(kAttnThreads, attn_min_blocks<T, NB>())
attn_res_fixed_kernel(const T *__restrict__ V, const float *__restrict__ w, T *__restrict__ h,
                      long long rows, int D, float eps) {
  using P = Piece<T>;
  constexpr int E = P::E;
  __shared__ float red[kAttnWarps][NB][2];
  __shared__ float alpha[NB];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npieces = D / E;
  const size_t stride = (size_t)rows * D;

  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const T *vr = V + (size_t)row * D;
    float dot[NB], ss[NB];
#pragma unroll
    for (int n = 0; n < NB; ++n) dot[n] = ss[n] = 0.f;
#pragma unroll 1
    for (int pc = tid; pc < npieces; pc += kAttnThreads) {
      float x[NB][E];
#pragma unroll
      for (int n = 0; n < NB; ++n) P::load(vr + (size_t)n * stride + (size_t)pc * E, x[n], Use::first);
      float wv[E];
      const float4 *wp = reinterpret_cast<const float4 *>(w + (size_t)pc * E);
#pragma unroll
      for (int i = 0; i < E / 4; ++i) {
        const float4 u = __ldg(wp + i);
        wv[4 * i] = u.x; wv[4 * i + 1] = u.y; wv[4 * i + 2] = u.z; wv[4 * i + 3] = u.w;
      }
#pragma unroll
      for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int e = 0; e < E; ++e) {
          dot[n] += wv[e] * x[n][e];
          ss[n] += x[n][e] * x[n][e];
        }
    }
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      float a = dot[n], b = ss[n];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
      }
      if (lane == 0) {
        red[warp][n][0] = a;
        red[warp][n][1] = b;
      }
    }
    __syncthreads();
    if (warp == 0) {
      float logit = -INFINITY;
      if (lane < NB) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int i = 0; i < kAttnWarps; ++i) {
          a += red[i][lane][0];
          b += red[i][lane][1];
        }
        logit = a * rsqrtf(b / (float)D + eps);
      }
      float m = logit;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      const float e = lane < NB ? __expf(logit - m) : 0.f;
      float sum = e;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane < NB) alpha[lane] = e / sum;
    }
    __syncthreads();
    if (tid == 0 && row + gridDim.x < rows) {
      // the first two blocks of this CTA's next row into L2 while pass 2 runs
      // from L2: HBM is otherwise idle for this CTA until that row's pass 1.
      // More than two (all nine: 124 us against 112) pushes rows that are
      // between their two reads out of L2.
      const T *nx = V + (size_t)(row + gridDim.x) * D;
      const uint32_t bytes = (uint32_t)min((size_t)D * sizeof(T), (size_t)32768);
#pragma unroll
      for (int n = 0; n < (NB < 2 ? NB : 2); ++n)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(nx + (size_t)n * stride),
                     "r"(bytes)
                     : "memory");
    }
    float al[NB];
#pragma unroll
    for (int n = 0; n < NB; ++n) al[n] = alpha[n];
    T *hr = h + (size_t)row * D;
#pragma unroll 1
    for (int pc = tid; pc < npieces; pc += kAttnThreads) {
      float x[NB][E];
#pragma unroll
      for (int n = 0; n < NB; ++n) P::load(vr + (size_t)n * stride + (size_t)pc * E, x[n], Use::last);
      float acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
      for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += al[n] * x[n][e];
      P::store(hr + (size_t)pc * E, acc);
    }
    __syncthreads();
  }
}

template <typename T, int NB>
void launch_fixed(const void *V, const float *w, void *h, long long rows, int D, float eps,
                  int grid, cudaStream_t stream) {
  attn_res_fixed_kernel<T, NB><<<grid, kAttnThreads, 0, stream>>>(
      static_cast<const T *>(V), w, static_cast<T *>(h), rows, D, eps);
}

template <typename T, int... Ns>
bool dispatch_fixed(int nb, std::integer_sequence<int, Ns...>, const void *V, const float *w,
                    void *h, long long rows, int D, float eps, int grid, cudaStream_t stream) {
  bool done = false;
  ((nb == Ns + 1 ? (launch_fixed<T, Ns + 1>(V, w, h, rows, D, eps, grid, stream), done = true)
                 : false),
   ...);
  return done;
}

}  // namespace

kda_status launch_attn_res(const void *V, int nb, const float *w, void *h, long long rows, int D,
                           kda_dtype dt, float eps, cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KDA_ERR_CUDA;
  const long long cap = (long long)sms * 16;
  const int grid = (int)(rows < cap ? rows : cap);
  const auto seq = std::make_integer_sequence<int, kFixedMax>{};
  const bool fixed = dt == KDA_BF16
                         ? dispatch_fixed<__nv_bfloat16>(nb, seq, V, w, h, rows, D, eps, grid, stream)
                         : dispatch_fixed<float>(nb, seq, V, w, h, rows, D, eps, grid, stream);
  if (fixed) return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
  if (dt == KDA_BF16)
    attn_res_kernel<__nv_bfloat16><<<grid, kAttnThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(V), nb, w, static_cast<__nv_bfloat16 *>(h), rows, D,
        eps);
  else
    attn_res_kernel<float><<<grid, kAttnThreads, 0, stream>>>(
        static_cast<const float *>(V), nb, w, static_cast<float *>(h), rows, D, eps);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda

extern "C" kda_status kda_attn_res(const void *V, int n_blocks, const float *w, void *h,
                                   long long rows, int D, kda_dtype dt, float eps,
                                   kda_stream_t stream) {
  using namespace kda;
  if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (rows < 0 || D <= 0 || n_blocks < 1 || !(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (n_blocks > kMaxBlocks || D % 8 != 0 || D > (1 << 20)) return KDA_ERR_UNSUPPORTED;
  if (rows == 0) return KDA_OK;
  if (!V || !w || !h) return KDA_ERR_INVALID_ARG;
  const auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(V) || !a16(w) || !a16(h)) return KDA_ERR_INVALID_ARG;
  return launch_attn_res(V, n_blocks, w, h, rows, D, dt, eps,
                         reinterpret_cast<cudaStream_t>(stream));
}
