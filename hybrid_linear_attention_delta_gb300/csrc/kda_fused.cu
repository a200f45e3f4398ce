// kda_fused.cu -- the layer around the KDA recurrence that a serving stack
// runs with it: a short causal convolution of the raw q, k, v channels, whose
// last inputs are kept per slot beside the matrix state, and the gated
// RMSNorm of the outputs.
//
// "Kimi K3 + vLLM: Inside the Day-0 Production Integration": a KDA layer keeps
// "a short causal convolution state" beside its matrix state ("Kimi Delta
// Attention: When Prefix Caching Meets Recurrent State"), and its fused decode
// kernel folds the causal convolution, the recurrent state update, the gating
// and the RMSNorm into one launch ("Separate Prefill/Decode Code Paths"); the
// vLLM recipe page for Kimi-K3 fuses the output RMSNorm and its sigmoid gate
// into one kernel.  Per token t and head h, with W = 4 taps per channel:
//     [q~ | k~ | v~]_t = act(sum_i w[c][i] x[t - (W-1) + i][c])   (raw x, causal)
//     q = q~ / |q~| / sqrt(dk),  k = k~ / |k~|,  v = v~             (then the recurrence)
//     y_t = o_t / sqrt(mean(o_t^2) + eps) * w_norm * sigmoid(gate_t)
// Decode runs all of it in one kernel (decode_fused_kernel).  Prefill runs it
// around the chunked kernels: conv_prefill_kernel writes q, k, v for the
// batch, conv_state_kernel the new convolution states, and rms_gate_kernel
// turns the prefill's outputs into y.  Reductions (L2 norms, RMS) run in a
// fixed order: results are deterministic.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kConvTile = 16;     // tokens per CTA of the prefill convolution
constexpr int kMaxConvC = 384;    // channels of a head: 2 dk + dv <= 384

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }
__device__ __forceinline__ float act_f(float y, int act) {
  return act == 1 ? y / (1.f + expf(-y)) : y;
}

template <typename T>
__device__ __forceinline__ float raw_input(const FusedParams &f, int64_t t, int H, int h, int dk,
                                           int dv, int c) {
  if (c < dk) return to_f32(static_cast<const T *>(f.xq)[(t * H + h) * dk + c]);
  if (c < 2 * dk) return to_f32(static_cast<const T *>(f.xk)[(t * H + h) * dk + c - dk]);
  return to_f32(static_cast<const T *>(f.xv)[(t * H + h) * dv + c - 2 * dk]);
}

// Sequence of packed token t: the largest b with cu[b] <= t (cu validated by
// the plan kernel; empty sequences are skipped by taking the largest).
__device__ __forceinline__ int seq_of(const int32_t *cu, int B, int64_t t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One CTA: kConvTile packed tokens x one head; thread c: channel c of the
// head's 2 dk + dv.  The tile's raw inputs are loaded together first; the
// convolution then runs token by token with the channel's last inputs in
// registers.  |q~| and |k~| of each token are reduced by one warp per (token,
// part) in a fixed order (deterministic).  Writes q, k, v (the recurrence's
// inputs) for tokens of sequences the plan accepted.
template <typename T>
__global__ void __launch_bounds__(kMaxConvC) conv_prefill_kernel(PrefillPlan p, FusedParams f) {
  const int c = threadIdx.x, h = blockIdx.y, H = p.H, dk = p.dk, dv = p.dv;
  const int C = 2 * dk + dv;
  const int64_t t0 = (int64_t)blockIdx.x * kConvTile;
  const int n = (int)min((int64_t)kConvTile, (int64_t)p.T_total - t0);
  __shared__ float ss[kConvTile][256];     // squares of the q and k channels
  __shared__ float sinv[2][kConvTile];     // 1 / |q~|, 1 / |k~| per token
  __shared__ int sb0;
  if (c == 0) sb0 = seq_of(p.cu_seqlens, p.B, t0);
  float xs[kConvTile];
  if (c < C) {
#pragma unroll
    for (int tt = 0; tt < kConvTile; ++tt)
      xs[tt] = tt < n ? raw_input<T>(f, t0 + tt, H, h, dk, dv, c) : 0.f;
  }
  __syncthreads();
  float y[kConvTile];
  int ok_mask = 0;  // bit tt: token t0 + tt belongs to an accepted sequence
  if (c < C) {
    float w[kConvW];
#pragma unroll
    for (int i = 0; i < kConvW; ++i) w[i] = f.conv_w[((int64_t)h * C + c) * kConvW + i];
    int b = sb0;
    int64_t start = p.cu_seqlens[b], end = p.cu_seqlens[b + 1];
    int ok = p.meta[b].ok;
    float hist[kConvW - 1];
    // the kConvW - 1 raw inputs before token t of sequence b, from the
    // sequence itself or from its starting convolution state
    auto init_hist = [&](int64_t t) {
      const int src = p.meta[b].src;
      const T *cp = static_cast<const T *>(f.conv_pool);
#pragma unroll
      for (int i = 0; i < kConvW - 1; ++i) {
        const int64_t pos = t - start - (kConvW - 1) + i;
        if (pos >= 0)
          hist[i] = raw_input<T>(f, start + pos, H, h, dk, dv, c);
        else if (src >= 0)
          hist[i] = to_f32(cp[(((int64_t)src * H + h) * C + c) * (kConvW - 1) +
                              (kConvW - 1 + pos)]);
        else
          hist[i] = 0.f;
      }
    };
    init_hist(t0);
#pragma unroll
    for (int tt = 0; tt < kConvTile; ++tt) {
      y[tt] = 0.f;
      if (tt >= n) continue;
      const int64_t t = t0 + tt;
      if (t >= end) {  // the next sequence (skipping empty ones) starts here
        while (t >= end) {
          ++b;
          start = p.cu_seqlens[b];
          end = p.cu_seqlens[b + 1];
        }
        ok = p.meta[b].ok;
        init_hist(t);
      }
      float acc = w[kConvW - 1] * xs[tt];
#pragma unroll
      for (int i = 0; i < kConvW - 1; ++i) acc = fmaf(w[i], hist[i], acc);
#pragma unroll
      for (int i = 0; i + 1 < kConvW - 1; ++i) hist[i] = hist[i + 1];
      hist[kConvW - 2] = xs[tt];
      y[tt] = act_f(acc, f.act);
      if (ok) ok_mask |= 1 << tt;
      if (c < 2 * dk) ss[tt][c] = y[tt] * y[tt];
    }
  }
  __syncthreads();
  // |q~| and |k~| of each token: warp w takes (token, part) pairs w, w + warps,
  // ...; lane i sums channels i, i + 32, ... of the part, then a fixed tree
  {
    const int warp = c >> 5, lane = c & 31, nwarps = blockDim.x >> 5;
    for (int pr = warp; pr < 2 * n; pr += nwarps) {
      const int tt = pr >> 1, part = pr & 1;
      float sum = 0.f;
      for (int i = lane; i < dk; i += 32) sum += ss[tt][part * dk + i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) sinv[part][tt] = sum > 0.f ? rsqrtf(sum) : 0.f;
    }
  }
  __syncthreads();
  if (c >= C) return;
  const float qscale = rsqrtf((float)dk);
#pragma unroll
  for (int tt = 0; tt < kConvTile; ++tt) {
    if (!(ok_mask >> tt & 1)) continue;
    const int64_t t = t0 + tt;
    if (c < dk)
      static_cast<T *>(const_cast<void *>(p.q))[(t * H + h) * dk + c] =
          from_f32<T>(y[tt] * sinv[0][tt] * qscale);
    else if (c < 2 * dk)
      static_cast<T *>(const_cast<void *>(p.k))[(t * H + h) * dk + c - dk] =
          from_f32<T>(y[tt] * sinv[1][tt]);
    else
      static_cast<T *>(const_cast<void *>(p.v))[(t * H + h) * dv + c - 2 * dk] = from_f32<T>(y[tt]);
  }
}

// One CTA per (sequence, head); thread c: channel c.  The new state of a
// channel is the last kConvW - 1 raw inputs of [old state; sequence], read
// before anything is written (so src == dst extends in place).
template <typename T>
__global__ void __launch_bounds__(kMaxConvC) conv_state_kernel(PrefillPlan p, FusedParams f) {
  const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x, H = p.H, dk = p.dk, dv = p.dv;
  const int C = 2 * dk + dv;
  const SeqMeta m = p.meta[b];
  if (!m.ok || c >= C) return;
  T *cp = static_cast<T *>(f.conv_pool);
  float ns[kConvW - 1];
#pragma unroll
  for (int i = 0; i < kConvW - 1; ++i) {
    const int64_t pos = (int64_t)m.len - (kConvW - 1) + i;
    if (pos >= 0)
      ns[i] = raw_input<T>(f, (int64_t)m.tok0 + pos, H, h, dk, dv, c);
    else if (m.src >= 0)
      ns[i] = to_f32(cp[(((int64_t)m.src * H + h) * C + c) * (kConvW - 1) + (kConvW - 1 + pos)]);
    else
      ns[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < kConvW - 1; ++i)
    cp[(((int64_t)m.dst * H + h) * C + c) * (kConvW - 1) + i] = from_f32<T>(ns[i]);
}

// y = o / rms(o) * w * sigmoid(gate) per (token, head) row of dv outputs.
// One warp takes kRmsRows consecutive rows and issues all their loads (o,
// gate and the row's sequence check) before it reduces; rows of sequences
// the plan did not accept are not written.
constexpr int kRmsRows = 4;

template <typename T>
__global__ void __launch_bounds__(256) rms_gate_kernel(PrefillPlan p, FusedParams f, const T *o,
                                                       T *out) {
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * kRmsRows;
  const int H = p.H, dv = p.dv;
  const int64_t rows = (int64_t)p.T_total * H;
  const T *gate = static_cast<const T *>(f.gate);
  float v[kRmsRows][4], gt[kRmsRows][4];
  int ok[kRmsRows];
#pragma unroll
  for (int r = 0; r < kRmsRows; ++r) {
    const int64_t row = row0 + r;
    ok[r] = row < rows;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = lane + 32 * e;
      const bool in = ok[r] && j < dv;
      v[r][e] = in ? to_f32(o[row * dv + j]) : 0.f;
      gt[r][e] = in ? to_f32(gate[row * dv + j]) : 0.f;
    }
    if (ok[r]) ok[r] = p.meta[seq_of(p.cu_seqlens, p.B, row / H)].ok;
  }
#pragma unroll
  for (int r = 0; r < kRmsRows; ++r) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) ss = fmaf(v[r][e], v[r][e], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (!ok[r]) continue;
    const float rr = rsqrtf(ss / (float)dv + f.eps);
    const int64_t row = row0 + r;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = lane + 32 * e;
      if (j < dv) out[row * dv + j] = from_f32<T>(v[r][e] * rr * f.norm_w[j] * sigmoid_f(gt[r][e]));
    }
  }
}

// ------------------------------------------------------------------ decode
// One CTA of 256 threads per (sequence, head), dk = dv = 128; the state
// layout of the 128 x 128 decode kernels (warp w: rows [16 w, +16), lane l:
// columns [4 l, +4)), read once and written once.  Per token: the
// convolution of the 384 raw channels (thread c and c + 256), the L2
// normalisation of q and k, their rounding to the call's element type (the
// type every call's recurrence takes them in), the recurrence step, the gated
// RMSNorm of the output; the channel's last three raw inputs stay in shared memory and go
// back to the slot's convolution state at the end.
constexpr int kD = 128;
constexpr int kDecThreads = 256;
constexpr int kRows = kD / (kDecThreads / 32);  // 16
constexpr int kC3 = 3 * kD;                     // channels q | k | v

template <typename T>
__global__ void __launch_bounds__(kDecThreads, 2) decode_fused_kernel(DecodePlan p, FusedParams f) {
  const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
  const int H = p.H;
  const int n = blockIdx.x / H, h = blockIdx.x % H;
  __shared__ int s_slot;
  __shared__ float hist[kC3][kConvW - 1];
  __shared__ float cw[kC3][kConvW];
  __shared__ __align__(16) float sq[kD], sk[kD], sv[kD], sa[kD], sg[kD];
  __shared__ __align__(16) float su[kD], sy[kD];
  __shared__ __align__(16) float redx[kDecThreads / 32][kD], redy[kDecThreads / 32][kD];
  __shared__ float red[kDecThreads / 32];
  __shared__ float sbeta;

  if (tid == 0) {
    int slot = p.slot_ids[n];
    if (slot < 0 || slot >= p.n_slots) {
      raise_error(p.err, ERR_BAD_SLOT);
      slot = -1;
    } else if (!claim_state(p.claims, ((int64_t)slot * H + h) * kClaimsPerState, p.epoch)) {
      raise_error(p.err, ERR_DUP_SLOT);
      slot = -1;
    }
    s_slot = slot;
  }
  __syncthreads();
  const int slot = s_slot;
  if (slot < 0) return;

  T *cpool = static_cast<T *>(f.conv_pool) + ((int64_t)slot * H + h) * kC3 * (kConvW - 1);
  for (int c = tid; c < kC3; c += kDecThreads) {
#pragma unroll
    for (int i = 0; i < kConvW - 1; ++i) hist[c][i] = to_f32(cpool[c * (kConvW - 1) + i]);
#pragma unroll
    for (int i = 0; i < kConvW; ++i) cw[c][i] = f.conv_w[((int64_t)h * kC3 + c) * kConvW + i];
  }
  const int64_t kStateElems = (int64_t)kD * kD;
  float *state = p.pool + ((int64_t)slot * H + h) * kStateElems;
  float4 s[kRows];
#pragma unroll
  for (int m = 0; m < kRows; ++m)
    s[m] = __ldcs(reinterpret_cast<const float4 *>(state + (w * kRows + m) * kD) + l);
  const T *g = (const T *)p.g, *beta = (const T *)p.beta, *gate = (const T *)f.gate;
  T *out = (T *)p.out;
  const float nw = tid < kD ? f.norm_w[tid] : 0.f;
  const float qscale = rsqrtf((float)kD);
  __syncthreads();

  for (int j = 0; j < p.n_tok; ++j) {
    const int64_t t = (int64_t)n * p.n_tok + j, row = t * H + h;
    // convolution of the 384 channels: thread tid takes channel tid (q or k)
    // and, for tid < 128, channel 256 + tid (v)
    float ysq = 0.f;
    for (int c = tid; c < kC3; c += kDecThreads) {
      const float x = raw_input<T>(f, t, H, h, kD, kD, c);
      float acc = cw[c][kConvW - 1] * x;
#pragma unroll
      for (int i = 0; i < kConvW - 1; ++i) acc = fmaf(cw[c][i], hist[c][i], acc);
#pragma unroll
      for (int i = 0; i + 1 < kConvW - 1; ++i) hist[c][i] = hist[c][i + 1];
      hist[c][kConvW - 2] = x;
      const float y = act_f(acc, f.act);
      if (c < kD) { sq[c] = y; ysq = y * y; }
      else if (c < 2 * kD) { sk[c - kD] = y; ysq = y * y; }
      else sv[c - 2 * kD] = y;
    }
    if (tid < kD) {
      sa[tid] = expf(to_f32(g[row * kD + tid]));
      sg[tid] = sigmoid_f(to_f32(gate[row * kD + tid]));
    }
    if (tid == 0) sbeta = to_f32(beta[row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ysq += __shfl_xor_sync(0xffffffffu, ysq, off);
    if (l == 0) red[w] = ysq;  // warps 0-3: |q~|^2 partials, 4-7: |k~|^2
    __syncthreads();
    {  // the recurrence takes q, k, v in the call's element type (as the prefill does)
      const float qn = (red[0] + red[1]) + (red[2] + red[3]);
      const float kn = (red[4] + red[5]) + (red[6] + red[7]);
      if (tid < kD) {
        sq[tid] = to_f32(from_f32<T>(sq[tid] * (qn > 0.f ? rsqrtf(qn) : 0.f) * qscale));
        sv[tid] = to_f32(from_f32<T>(sv[tid]));
      } else {
        sk[tid - kD] = to_f32(from_f32<T>(sk[tid - kD] * (kn > 0.f ? rsqrtf(kn) : 0.f)));
      }
    }
    __syncthreads();
    // the recurrence step of the 128 x 128 decode kernels
    float kq = 0.f;
    if (tid < kD) kq = sq[tid] * sk[tid];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
    float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f), y4 = x4;
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
      const int i = w * kRows + m;
      const float ai = sa[i], ki = sk[i], qi = sq[i];
      s[m].x *= ai; s[m].y *= ai; s[m].z *= ai; s[m].w *= ai;
      x4.x = fmaf(ki, s[m].x, x4.x); x4.y = fmaf(ki, s[m].y, x4.y);
      x4.z = fmaf(ki, s[m].z, x4.z); x4.w = fmaf(ki, s[m].w, x4.w);
      y4.x = fmaf(qi, s[m].x, y4.x); y4.y = fmaf(qi, s[m].y, y4.y);
      y4.z = fmaf(qi, s[m].z, y4.z); y4.w = fmaf(qi, s[m].w, y4.w);
    }
    *reinterpret_cast<float4 *>(&redx[w][4 * l]) = x4;
    *reinterpret_cast<float4 *>(&redy[w][4 * l]) = y4;
    __syncthreads();  // (the q . k partials of warps 0-3 go through red as well)
    if (l == 0 && w < 4) red[w] = kq;
    if (tid < kD) {
      float xs = 0.f;
#pragma unroll
      for (int ww = 0; ww < kDecThreads / 32; ++ww) xs += redx[ww][tid];
      su[tid] = sbeta * (sv[tid] - xs);
    } else {
      float ys = 0.f;
#pragma unroll
      for (int ww = 0; ww < kDecThreads / 32; ++ww) ys += redy[ww][tid - kD];
      sy[tid - kD] = ys;
    }
    __syncthreads();
    // output o = y + u (k . q), then its RMSNorm and gate
    float o = 0.f;
    if (tid < kD) o = fmaf(su[tid], (red[0] + red[1]) + (red[2] + red[3]), sy[tid]);
    float osq = o * o;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) osq += __shfl_xor_sync(0xffffffffu, osq, off);
    const float4 u4 = *reinterpret_cast<const float4 *>(&su[4 * l]);
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
      const float ki = sk[w * kRows + m];
      s[m].x = fmaf(ki, u4.x, s[m].x); s[m].y = fmaf(ki, u4.y, s[m].y);
      s[m].z = fmaf(ki, u4.z, s[m].z); s[m].w = fmaf(ki, u4.w, s[m].w);
    }
    if (p.per_tok) {
      float *pt = p.per_tok + (t * H + h) * kStateElems;
#pragma unroll
      for (int m = 0; m < kRows; ++m)
        __stcs(reinterpret_cast<float4 *>(pt + (w * kRows + m) * kD) + l, s[m]);
    }
    __syncthreads();  // every read of red (k . q) is done
    if (l == 0 && w < 4) red[w] = osq;
    __syncthreads();
    if (tid < kD) {
      const float r = rsqrtf(((red[0] + red[1]) + (red[2] + red[3])) / (float)kD + f.eps);
      out[row * kD + tid] = from_f32<T>(o * r * nw * sg[tid]);
    }
    __syncthreads();  // the next token's staging overwrites sq, sk, red
  }

#pragma unroll
  for (int m = 0; m < kRows; ++m)
    __stcs(reinterpret_cast<float4 *>(state + (w * kRows + m) * kD) + l, s[m]);
  for (int c = tid; c < kC3; c += kDecThreads) {
#pragma unroll
    for (int i = 0; i < kConvW - 1; ++i) cpool[c * (kConvW - 1) + i] = from_f32<T>(hist[c][i]);
  }
}

}  // namespace

cudaError_t launch_conv_prefill(const PrefillPlan &p, const FusedParams &f) {
  if (p.T_total == 0) return cudaSuccess;
  const int C = 2 * p.dk + p.dv;
  dim3 grid((unsigned)((p.T_total + kConvTile - 1) / kConvTile), p.H);
  const int threads = (C + 31) / 32 * 32;
  if (p.dtype == KDA_BF16)
    conv_prefill_kernel<__nv_bfloat16><<<grid, threads, 0, p.stream>>>(p, f);
  else
    conv_prefill_kernel<float><<<grid, threads, 0, p.stream>>>(p, f);
  return cudaGetLastError();
}

cudaError_t launch_conv_state(const PrefillPlan &p, const FusedParams &f) {
  if (p.B == 0) return cudaSuccess;
  const int C = 2 * p.dk + p.dv;
  dim3 grid(p.B, p.H);
  const int threads = (C + 31) / 32 * 32;
  if (p.dtype == KDA_BF16)
    conv_state_kernel<__nv_bfloat16><<<grid, threads, 0, p.stream>>>(p, f);
  else
    conv_state_kernel<float><<<grid, threads, 0, p.stream>>>(p, f);
  return cudaGetLastError();
}

cudaError_t launch_rms_gate(const PrefillPlan &p, const FusedParams &f, const void *o, void *out) {
  const int64_t rows = (int64_t)p.T_total * p.H;
  if (rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + 8 * kRmsRows - 1) / (8 * kRmsRows));
  if (p.dtype == KDA_BF16)
    rms_gate_kernel<__nv_bfloat16><<<grid, 256, 0, p.stream>>>(
        p, f, static_cast<const __nv_bfloat16 *>(o), static_cast<__nv_bfloat16 *>(out));
  else
    rms_gate_kernel<float><<<grid, 256, 0, p.stream>>>(p, f, static_cast<const float *>(o),
                                                       static_cast<float *>(out));
  return cudaGetLastError();
}

cudaError_t launch_decode_fused(const DecodePlan &p, const FusedParams &f) {
  if (p.N == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((int64_t)p.N * p.H);
  if (p.dtype == KDA_BF16)
    decode_fused_kernel<__nv_bfloat16><<<grid, kDecThreads, 0, p.stream>>>(p, f);
  else
    decode_fused_kernel<float><<<grid, kDecThreads, 0, p.stream>>>(p, f);
  return cudaGetLastError();
}

}  // namespace kda
