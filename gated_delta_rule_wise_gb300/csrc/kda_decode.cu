// kda_decode.cu -- single-token recurrent decode step of the gated delta rule.
//
// For each of N x H independent states S [dk][dv] (float32, in place):
//   S' = Diag(a) S                   a = exp(-exp(log_alpha)), per key channel
//   u  = beta (v - S'^T k)
//   S  = S' + k u^T
//   o  = S^T q = S'^T q + (k . q) u
// ("22,580: From GPT-2 to Kimi K3" (yichencityu.github.io), section 5.2, the
// decode-time forward with a cached state; the per-channel decay of
// "22580: From GPT-2 to Kimi K3, Explained" (lukebest.github.io), "KDA
// (per-channel alpha)", applied before the read.)
//
// The step is HBM-bound (about 0.9 flop per byte of state), so the kernel is
// one streaming pass: each CTA owns a block of up to 64 value columns of one
// state (the columns never mix: S'^T k, S'^T q and u are per column), loads
// it into registers with 128-bit streaming loads, forms the two column
// reductions and writes S' + k u^T back with 128-bit streaming stores.  One
// read and one write of the state, nothing else touches HBM in bulk; column
// blocks keep several small CTAs per SM in flight.
#include "kda_launch.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeCols = 64;  // value columns per CTA (at most)

template <int DK, int DV, typename TI>
__global__ void __launch_bounds__(kDecodeThreads, 4)
decode_step_kernel(const TI *__restrict__ q, const TI *__restrict__ k,
                   const TI *__restrict__ v, const float *__restrict__ beta,
                   const float *__restrict__ log_alpha, int alpha_mode,
                   float *__restrict__ S, TI *__restrict__ o) {
  constexpr int NT = kDecodeThreads;
  constexpr int DVB = DV < kDecodeCols ? DV : kDecodeCols;  // this CTA's value columns
  constexpr int NBLK = DV / DVB;
  constexpr int C4 = DVB / 4;              // float4 column groups per row
  constexpr int G = NT / C4;               // threads that share a column group
  constexpr int PER = (DK + G - 1) / G;    // float4s held per thread
  static_assert(NT % C4 == 0, "column groups must tile the block");

  __shared__ float s_k[DK], s_q[DK], s_a[DK];
  __shared__ float4 red_k[NT], red_q[NT];
  __shared__ __align__(16) float s_u[DVB];
  __shared__ float s_kq;

  const int sid = blockIdx.x / NBLK;  // state index n * H + h
  const int j0 = (blockIdx.x % NBLK) * DVB;
  const int tid = threadIdx.x;
  const int c4 = tid % C4;
  const int r0 = tid / C4;
  float *Sp = S + (size_t)sid * DK * DV + j0;

  // Issue every state load first: the whole 64 KiB (at 128 x 128) is in
  // flight before anything waits on it.
  float4 s[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int r = r0 + j * G;
    if (r < DK) s[j] = __ldcs(reinterpret_cast<const float4 *>(Sp + (size_t)r * DV) + c4);
  }

  for (int i = tid; i < DK; i += NT) {
    s_k[i] = Io<TI>::ld(k + (size_t)sid * DK + i);
    s_q[i] = Io<TI>::ld(q + (size_t)sid * DK + i);
    float a = 1.0f;
    if (alpha_mode == KDA_ALPHA_CHANNEL)
      a = decay_of(log_alpha[(size_t)sid * DK + i]);
    else if (alpha_mode == KDA_ALPHA_SCALAR)
      a = decay_of(log_alpha[sid]);
    s_a[i] = a;
  }
  __syncthreads();

  if (tid < 32) {  // k . q, read after the next barrier
    float acc = 0.f;
    for (int i = tid; i < DK; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (tid == 0) s_kq = acc;
  }

  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int r = r0 + j * G;
    if (r < DK) {
      const float a = s_a[r], kr = s_k[r], qr = s_q[r];
      s[j].x *= a; s[j].y *= a; s[j].z *= a; s[j].w *= a;
      pk.x += kr * s[j].x; pk.y += kr * s[j].y; pk.z += kr * s[j].z; pk.w += kr * s[j].w;
      pq.x += qr * s[j].x; pq.y += qr * s[j].y; pq.z += qr * s[j].z; pq.w += qr * s[j].w;
    }
  }
  red_k[tid] = pk;
  red_q[tid] = pq;
  __syncthreads();

  if (tid < C4) {
    float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sq = sk;
#pragma unroll 8
    for (int g = 0; g < G; ++g) {
      const float4 a = red_k[g * C4 + tid], b = red_q[g * C4 + tid];
      sk.x += a.x; sk.y += a.y; sk.z += a.z; sk.w += a.w;
      sq.x += b.x; sq.y += b.y; sq.z += b.z; sq.w += b.w;
    }
    const float bt = beta[sid], kq = s_kq;
    const float skv[4] = {sk.x, sk.y, sk.z, sk.w};
    const float sqv[4] = {sq.x, sq.y, sq.z, sq.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = tid * 4 + e;
      const float u = bt * (Io<TI>::ld(v + (size_t)sid * DV + j0 + col) - skv[e]);
      s_u[col] = u;
      Io<TI>::st(o + (size_t)sid * DV + j0 + col, sqv[e] + kq * u);
    }
  }
  __syncthreads();

  const float4 u4 = reinterpret_cast<const float4 *>(s_u)[c4];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int r = r0 + j * G;
    if (r < DK) {
      const float kr = s_k[r];
      float4 x = s[j];
      x.x += kr * u4.x; x.y += kr * u4.y; x.z += kr * u4.z; x.w += kr * u4.w;
      __stcs(reinterpret_cast<float4 *>(Sp + (size_t)r * DV) + c4, x);
    }
  }
}

template <int DK, typename TI>
kda_status launch_dk(const void *q, const void *k, const void *v, const float *beta,
                     const float *la, float *S, void *o, int NH, int dv, int am,
                     cudaStream_t st) {
  const int nblk = dv < kDecodeCols ? 1 : dv / kDecodeCols;
  if ((long long)NH * nblk > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
  const dim3 grid(NH * nblk), block(kDecodeThreads);
  const TI *qq = static_cast<const TI *>(q), *kk = static_cast<const TI *>(k),
           *vv = static_cast<const TI *>(v);
  TI *oo = static_cast<TI *>(o);
  switch (dv) {
    case 16: decode_step_kernel<DK, 16, TI><<<grid, block, 0, st>>>(qq, kk, vv, beta, la, am, S, oo); break;
    case 32: decode_step_kernel<DK, 32, TI><<<grid, block, 0, st>>>(qq, kk, vv, beta, la, am, S, oo); break;
    case 64: decode_step_kernel<DK, 64, TI><<<grid, block, 0, st>>>(qq, kk, vv, beta, la, am, S, oo); break;
    case 128: decode_step_kernel<DK, 128, TI><<<grid, block, 0, st>>>(qq, kk, vv, beta, la, am, S, oo); break;
    default: return KDA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

template <typename TI>
kda_status launch_t(const void *q, const void *k, const void *v, const float *beta,
                    const float *la, float *S, void *o, int NH, int dk, int dv, int am,
                    cudaStream_t st) {
  switch (dk) {
    case 16: return launch_dk<16, TI>(q, k, v, beta, la, S, o, NH, dv, am, st);
    case 32: return launch_dk<32, TI>(q, k, v, beta, la, S, o, NH, dv, am, st);
    case 64: return launch_dk<64, TI>(q, k, v, beta, la, S, o, NH, dv, am, st);
    case 128: return launch_dk<128, TI>(q, k, v, beta, la, S, o, NH, dv, am, st);
    default: return KDA_ERR_UNSUPPORTED;
  }
}

}  // namespace

kda_status launch_decode(const void *q, const void *k, const void *v, const float *beta,
                         const float *log_alpha, float *S, void *o, int N, int H, int dk,
                         int dv, kda_dtype dt, kda_alpha_mode am, cudaStream_t stream) {
  const long long NH = (long long)N * H;
  if (NH == 0) return KDA_OK;
  if (NH > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
  if (dt == KDA_BF16)
    return launch_t<__nv_bfloat16>(q, k, v, beta, log_alpha, S, o, (int)NH, dk, dv, am, stream);
  return launch_t<float>(q, k, v, beta, log_alpha, S, o, (int)NH, dk, dv, am, stream);
}

}  // namespace kda
