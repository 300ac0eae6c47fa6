// kda_host.cu -- kda_chunk_fwd with its inputs and outputs in host memory.
//
// The chunked prefill of a long sequence reads several bytes per token from
// HBM, but a caller whose q, k, v, beta and log_alpha sit in host memory must
// first move them over the host link, which is far slower than the kernels.
// This entry point cuts the work into pipeline steps and runs, for
// consecutive steps, the host -> device copy of step s + 1, the prefill of
// step s and the device -> host copy of step s - 1 at the same time: copy-in
// and copy-out on two streams of their own, the prefill on the caller's
// stream.  A step's inputs and outputs live in one of two staging slots of
// the caller's device buffer; the per-chunk workspace is shared by all steps
// (their prefills run one after another on the caller's stream).
//
// Steps are either segments of the sequence (the default: every (batch,
// head) pair, a chunk-aligned sixteenth of T; the state leaves one segment as
// hT and enters the next as h0, in float32, so the result is the one-call
// result bit for bit) or groups of (batch, head) pairs over all of T.  With
// segments the work left after the last copy-in is one segment's prefill and
// copy-out, not one group's whole-sequence scan.
#include <stdint.h>

#include <vector>

#include "kda_launch.cuh"

namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Bytes of each tensor for one (batch, head) pair.
struct PerHead {
  size_t q, v, beta, la, state, o;
};
PerHead per_head(int T, int dk, int dv, kda_dtype dt, kda_alpha_mode am) {
  const size_t es = dt == KDA_BF16 ? 2 : 4;
  PerHead p;
  p.q = (size_t)T * dk * es;  // q and k
  p.v = (size_t)T * dv * es;
  p.beta = (size_t)T * 4;
  p.la = am == KDA_ALPHA_CHANNEL ? (size_t)T * dk * 4 : (am == KDA_ALPHA_SCALAR ? (size_t)T * 4 : 0);
  p.state = (size_t)dk * dv * 4;  // h0 and hT
  p.o = p.v;
  return p;
}

// Layout of the device buffer for groups of G pairs: workspace, then two slots.
struct Layout {
  size_t ws, q, k, v, beta, la, h0, o, hT, slot, total;
};
Layout layout(const PerHead &p, int G, size_t ws_bytes) {
  Layout L;
  L.ws = up(ws_bytes);
  size_t off = 0;
  L.q = off;    off += up(G * p.q);
  L.k = off;    off += up(G * p.q);
  L.v = off;    off += up(G * p.v);
  L.beta = off; off += up(G * p.beta);
  L.la = off;   off += up(G * p.la);
  L.h0 = off;   off += up(G * p.state);
  L.o = off;    off += up(G * p.o);
  L.hT = off;   off += up(G * p.state);
  L.slot = off;
  L.total = L.ws + 2 * L.slot;
  return L;
}

// Segment mode: a chunk-aligned sixteenth of the sequence per step.
constexpr int kSegments = 16;
int seg_len(int T, int C) {
  const int t = (T + kSegments - 1) / kSegments;
  const int c = C > 0 ? C : 1;
  const int l = (t + c - 1) / c * c;
  return l > 0 ? l : c;
}
// Device buffer of the segment mode: workspace, the carried state, two slots.
struct SegLayout {
  size_t ws, state, q, k, v, beta, la, o, slot, total;
};
SegLayout seg_layout(const PerHead &p1, int BH, int Tl, int T, size_t ws_bytes) {
  // p1: per-head bytes for the whole sequence; a slot holds Tl tokens of every head
  SegLayout L;
  L.ws = up(ws_bytes);
  L.state = up((size_t)BH * p1.state);
  const size_t tq = T > 0 ? p1.q / T : 0, tv = T > 0 ? p1.v / T : 0;
  const size_t tb = T > 0 ? p1.beta / T : 0, tl = T > 0 ? p1.la / T : 0;
  size_t off = 0;
  L.q = off;    off += up((size_t)BH * Tl * tq);
  L.k = off;    off += up((size_t)BH * Tl * tq);
  L.v = off;    off += up((size_t)BH * Tl * tv);
  L.beta = off; off += up((size_t)BH * Tl * tb);
  L.la = off;   off += up((size_t)BH * Tl * tl);
  L.o = off;    off += up((size_t)BH * Tl * tv);
  L.slot = off;
  L.total = L.ws + L.state + 2 * L.slot;
  return L;
}

int group_of(int BH, int group_heads) {
  if (group_heads > 0) return group_heads < BH ? group_heads : BH;
  const int g = (BH + 7) / 8;  // eight groups by default
  return g > 0 ? g : 1;
}

// Streams and events of one call, released when the call returns (the CUDA
// runtime frees them once the work queued on them has finished).
struct Resources {
  cudaStream_t in = nullptr, out = nullptr;
  std::vector<cudaEvent_t> events;
  ~Resources() {
    for (cudaEvent_t e : events) cudaEventDestroy(e);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
  }
  cudaEvent_t make() {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    events.push_back(e);
    return e;
  }
};

}  // namespace

extern "C" size_t kda_chunk_fwd_host_buffer_size(int B, int H, int T, int dk, int dv, int C,
                                                 kda_dtype dt, kda_alpha_mode am,
                                                 int group_heads) {
  if (B < 0 || H < 0 || group_heads < 0) return 0;
  const int BH = B * H;
  if (group_heads == 0 && T > 0) {  // segments of the sequence
    const int Tl = seg_len(T, C);
    const size_t ws = kda_chunk_fwd_workspace_size(1, BH, Tl, dk, dv, C, dt, am);
    if (ws == 0) return 0;
    return seg_layout(per_head(T, dk, dv, dt, am), BH, Tl, T, ws).total;
  }
  const int G = group_of(BH, group_heads);
  const size_t ws = kda_chunk_fwd_workspace_size(1, G, T, dk, dv, C, dt, am);
  if (ws == 0) return 0;
  return layout(per_head(T, dk, dv, dt, am), G, ws).total;
}

namespace {

// Segment mode of kda_chunk_fwd_host (arguments already checked; T > 0).
kda_status host_segments(const void *q, const void *k, const void *v, const float *beta,
                         const float *log_alpha, const float *h0, void *o, float *hT, int BH,
                         int T, int dk, int dv, int C, kda_dtype dt, kda_alpha_mode am,
                         uint8_t *base, cudaStream_t s) {
  const int Tl = seg_len(T, C);
  const int NS = (T + Tl - 1) / Tl;
  const PerHead p = per_head(T, dk, dv, dt, am);
  const size_t tq = p.q / T, tv = p.v / T, tb = p.beta / T, tla = p.la / T;  // bytes per token
  const size_t ws_bytes = kda_chunk_fwd_workspace_size(1, BH, Tl, dk, dv, C, dt, am);
  const SegLayout L = seg_layout(p, BH, Tl, T, ws_bytes);
  uint8_t *ws = base;
  float *state = reinterpret_cast<float *>(base + L.ws);

  Resources R;
  if (cudaStreamCreateWithFlags(&R.in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&R.out, cudaStreamNonBlocking) != cudaSuccess)
    return KDA_ERR_CUDA;
  cudaEvent_t start = R.make();
  if (!start || cudaEventRecord(start, s) != cudaSuccess ||
      cudaStreamWaitEvent(R.in, start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(R.out, start, 0) != cudaSuccess)
    return KDA_ERR_CUDA;
  // the initial state goes in ahead of the first segment (same stream)
  if (h0 && cudaMemcpyAsync(state, h0, (size_t)BH * p.state, cudaMemcpyHostToDevice, R.in) !=
                cudaSuccess)
    return KDA_ERR_CUDA;

  std::vector<cudaEvent_t> out_done(NS, nullptr);
  for (int sg = 0; sg < NS; ++sg) {
    const int t0 = sg * Tl;
    const int Ts = T - t0 < Tl ? T - t0 : Tl;
    uint8_t *slot = base + L.ws + L.state + (size_t)(sg & 1) * L.slot;
    cudaEvent_t in_done = R.make(), comp_done = R.make();
    out_done[sg] = R.make();
    if (!in_done || !comp_done || !out_done[sg]) return KDA_ERR_CUDA;

    // copy-in: tokens t0 .. t0 + Ts of every (batch, head) pair, one 2-D copy
    // per tensor (host rows T tokens apart, device rows Ts tokens apart),
    // after the copy-out of the segment that last used this slot
    if (sg >= 2 && cudaStreamWaitEvent(R.in, out_done[sg - 2], 0) != cudaSuccess)
      return KDA_ERR_CUDA;
    auto h2d = [&](size_t off, const void *src, size_t per_token) {
      return cudaMemcpy2DAsync(slot + off, Ts * per_token,
                               static_cast<const uint8_t *>(src) + (size_t)t0 * per_token,
                               (size_t)T * per_token, Ts * per_token, BH,
                               cudaMemcpyHostToDevice, R.in) == cudaSuccess;
    };
    bool ok = h2d(L.q, q, tq) && h2d(L.k, k, tq) && h2d(L.v, v, tv) && h2d(L.beta, beta, tb);
    if (ok && am != KDA_ALPHA_NONE) ok = h2d(L.la, log_alpha, tla);
    if (!ok || cudaEventRecord(in_done, R.in) != cudaSuccess) return KDA_ERR_CUDA;

    // prefill of the segment: the state enters as h0 and leaves as hT
    if (cudaStreamWaitEvent(s, in_done, 0) != cudaSuccess) return KDA_ERR_CUDA;
    const bool last = sg == NS - 1;
    const kda_status st = kda_chunk_fwd(
        slot + L.q, slot + L.k, slot + L.v, reinterpret_cast<const float *>(slot + L.beta),
        am != KDA_ALPHA_NONE ? reinterpret_cast<const float *>(slot + L.la) : nullptr,
        (sg > 0 || h0) ? state : nullptr, slot + L.o, (!last || hT) ? state : nullptr, 1, BH, Ts,
        dk, dv, C, dt, am, ws, ws_bytes, reinterpret_cast<kda_stream_t>(s));
    if (st != KDA_OK) return st;
    if (cudaEventRecord(comp_done, s) != cudaSuccess) return KDA_ERR_CUDA;

    // copy-out of the segment's o (and of the final state)
    if (cudaStreamWaitEvent(R.out, comp_done, 0) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaMemcpy2DAsync(static_cast<uint8_t *>(o) + (size_t)t0 * tv, (size_t)T * tv, slot + L.o,
                          Ts * tv, Ts * tv, BH, cudaMemcpyDeviceToHost, R.out) != cudaSuccess)
      return KDA_ERR_CUDA;
    if (last && hT &&
        cudaMemcpyAsync(hT, state, (size_t)BH * p.state, cudaMemcpyDeviceToHost, R.out) !=
            cudaSuccess)
      return KDA_ERR_CUDA;
    if (cudaEventRecord(out_done[sg], R.out) != cudaSuccess) return KDA_ERR_CUDA;
  }
  if (cudaStreamWaitEvent(s, out_done[NS - 1], 0) != cudaSuccess) return KDA_ERR_CUDA;
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v,
                                         const float *beta, const float *log_alpha,
                                         const float *h0, void *o, float *hT, int B, int H, int T,
                                         int dk, int dv, int C, kda_dtype dt, kda_alpha_mode am,
                                         int group_heads, void *dev_buffer, size_t dev_bytes,
                                         kda_stream_t stream) {
  if (B < 0 || H < 0 || T < 0 || group_heads < 0) return KDA_ERR_INVALID_ARG;
  const size_t need = kda_chunk_fwd_host_buffer_size(B, H, T, dk, dv, C, dt, am, group_heads);
  if (need == 0)  // invalid or unsupported: let the full check name which
    return kda_chunk_fwd(q, k, v, beta, log_alpha, h0, o, hT, B, H, T, dk, dv, C, dt, am,
                         reinterpret_cast<void *>(kAlign), 0, stream);
  const int BH = B * H;
  if (BH == 0) return KDA_OK;
  if (!q || !k || !v || !beta || !o || (am != KDA_ALPHA_NONE && !log_alpha) || !dev_buffer)
    return KDA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_buffer) & (kAlign - 1)) != 0 || dev_bytes < need)
    return KDA_ERR_INVALID_ARG;

  if (group_heads == 0 && T > 0)
    return host_segments(q, k, v, beta, log_alpha, h0, o, hT, BH, T, dk, dv, C, dt, am,
                         static_cast<uint8_t *>(dev_buffer), reinterpret_cast<cudaStream_t>(stream));

  const int G = group_of(BH, group_heads);
  const int NG = (BH + G - 1) / G;
  const PerHead p = per_head(T, dk, dv, dt, am);
  const size_t ws_bytes = kda_chunk_fwd_workspace_size(1, G, T, dk, dv, C, dt, am);
  const Layout L = layout(p, G, ws_bytes);
  uint8_t *base = static_cast<uint8_t *>(dev_buffer);
  uint8_t *ws = base;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  Resources R;
  if (cudaStreamCreateWithFlags(&R.in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&R.out, cudaStreamNonBlocking) != cudaSuccess)
    return KDA_ERR_CUDA;
  // Both copy streams start after the work already queued on the caller's stream.
  cudaEvent_t start = R.make();
  if (!start || cudaEventRecord(start, s) != cudaSuccess ||
      cudaStreamWaitEvent(R.in, start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(R.out, start, 0) != cudaSuccess)
    return KDA_ERR_CUDA;

  const auto *hq = static_cast<const uint8_t *>(q);
  const auto *hk = static_cast<const uint8_t *>(k);
  const auto *hv = static_cast<const uint8_t *>(v);
  const auto *hb = reinterpret_cast<const uint8_t *>(beta);
  const auto *hla = reinterpret_cast<const uint8_t *>(log_alpha);
  const auto *hh0 = reinterpret_cast<const uint8_t *>(h0);
  auto *ho = static_cast<uint8_t *>(o);
  auto *hhT = reinterpret_cast<uint8_t *>(hT);

  std::vector<cudaEvent_t> out_done(NG, nullptr);
  for (int g = 0; g < NG; ++g) {
    const int b0 = g * G;
    const int Gg = BH - b0 < G ? BH - b0 : G;
    uint8_t *slot = base + L.ws + (size_t)(g & 1) * L.slot;
    cudaEvent_t in_done = R.make(), comp_done = R.make();
    out_done[g] = R.make();
    if (!in_done || !comp_done || !out_done[g]) return KDA_ERR_CUDA;

    // copy-in: after the copy-out of the group that last used this slot
    if (g >= 2 && cudaStreamWaitEvent(R.in, out_done[g - 2], 0) != cudaSuccess) return KDA_ERR_CUDA;
    auto h2d = [&](size_t off, const uint8_t *src, size_t per) {
      return cudaMemcpyAsync(slot + off, src + (size_t)b0 * per, (size_t)Gg * per,
                             cudaMemcpyHostToDevice, R.in) == cudaSuccess;
    };
    bool ok = h2d(L.q, hq, p.q) && h2d(L.k, hk, p.q) && h2d(L.v, hv, p.v) &&
              h2d(L.beta, hb, p.beta);
    if (ok && am != KDA_ALPHA_NONE) ok = h2d(L.la, hla, p.la);
    if (ok && h0) ok = h2d(L.h0, hh0, p.state);
    if (!ok || cudaEventRecord(in_done, R.in) != cudaSuccess) return KDA_ERR_CUDA;

    // prefill of the group on the caller's stream
    if (cudaStreamWaitEvent(s, in_done, 0) != cudaSuccess) return KDA_ERR_CUDA;
    const kda_status st = kda_chunk_fwd(
        slot + L.q, slot + L.k, slot + L.v, reinterpret_cast<const float *>(slot + L.beta),
        am != KDA_ALPHA_NONE ? reinterpret_cast<const float *>(slot + L.la) : nullptr,
        h0 ? reinterpret_cast<const float *>(slot + L.h0) : nullptr, slot + L.o,
        hT ? reinterpret_cast<float *>(slot + L.hT) : nullptr, 1, Gg, T, dk, dv, C, dt, am, ws,
        ws_bytes, stream);
    if (st != KDA_OK) return st;
    if (cudaEventRecord(comp_done, s) != cudaSuccess) return KDA_ERR_CUDA;

    // copy-out
    if (cudaStreamWaitEvent(R.out, comp_done, 0) != cudaSuccess) return KDA_ERR_CUDA;
    if (T > 0 && cudaMemcpyAsync(ho + (size_t)b0 * p.o, slot + L.o, (size_t)Gg * p.o,
                                 cudaMemcpyDeviceToHost, R.out) != cudaSuccess)
      return KDA_ERR_CUDA;
    if (hT && cudaMemcpyAsync(hhT + (size_t)b0 * p.state, slot + L.hT, (size_t)Gg * p.state,
                              cudaMemcpyDeviceToHost, R.out) != cudaSuccess)
      return KDA_ERR_CUDA;
    if (cudaEventRecord(out_done[g], R.out) != cudaSuccess) return KDA_ERR_CUDA;
  }
  // the call completes on the caller's stream
  if (cudaStreamWaitEvent(s, out_done[NG - 1], 0) != cudaSuccess) return KDA_ERR_CUDA;
  return KDA_OK;
}
