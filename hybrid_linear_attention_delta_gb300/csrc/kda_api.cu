// kda_api.cu -- the extern "C" entry points of libkda.so (declared in
// include/kda.h): host-side argument checks, workspace carving, and the
// stream-ordered launches.  No device memory is allocated here.
#include <cstring>
#include <mutex>
#include <set>
#include <unordered_map>
#include <utility>

#include "kda_internal.cuh"

namespace {

thread_local int32_t g_last_launches = 0;

// Epochs are counted per workspace: every stamp a call leaves in a workspace
// (slot claims, rerun flags, cooperative ready / consumed flags) holds that
// call's epoch, and a later call on the same workspace must never reuse it.
// When a workspace's 32-bit count wraps, its stamp regions are zero-filled on
// the call's stream (no allocation) before epoch 1 is handed out again.
std::mutex g_epoch_mu;
std::unordered_map<const void *, uint32_t> g_epochs;

cudaError_t next_epoch(const kda_args *a, uint32_t *epoch) {
  bool wrapped = false;
  {
    std::lock_guard<std::mutex> lock(g_epoch_mu);
    uint32_t &count = g_epochs[a->workspace];
    if (++count == 0) {  // 0 marks "never stamped"
      count = 1;
      wrapped = true;
    }
    *epoch = count;
  }
  if (!wrapped) return cudaSuccess;
  // every stamp in the workspace may equal an epoch of the new cycle: clear
  // everything but the sticky error word (stream-ordered, nothing allocated)
  const size_t n = kda::WorkspaceLayout(a->B, a->H, a->n_slots).total;
  return n > 256 ? cudaMemsetAsync(static_cast<char *>(a->workspace) + 256, 0, n - 256,
                                   static_cast<cudaStream_t>(a->stream))
                 : cudaSuccess;
}

bool dim_ok(int32_t d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status check_common(const kda_args *a) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->dtype != KDA_F32 && a->dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (a->B < 0 || a->T_total < 0 || a->H <= 0 || a->n_slots <= 0) return KDA_ERR_INVALID_ARG;
  if (!dim_ok(a->dk) || !dim_ok(a->dv)) return KDA_ERR_UNSUPPORTED;
  if (!a->workspace || (reinterpret_cast<uintptr_t>(a->workspace) & 255u)) return KDA_ERR_INVALID_ARG;
  if (a->workspace_bytes < kda_workspace_bytes(a)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

kda_status check_tokens(const void *q, const void *k, const void *v, const void *g,
                        const void *beta, const void *out, int64_t T) {
  if (T == 0) return KDA_OK;
  const void *ps[] = {q, k, v, g, beta, out};
  for (const void *p : ps)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

kda_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

void record(void *ev, cudaStream_t s) {
  if (ev) cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

}  // namespace

namespace kda {

cudaError_t set_smem_limit_once(const void *func, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void *, int>> done;  // (function, device)
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({func, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({func, dev});
  return e;
}

}  // namespace kda

extern "C" {

size_t kda_workspace_bytes(const kda_args *a) {
  if (!a || a->B < 0 || a->H <= 0 || a->n_slots < 0) return 0;
  return kda::WorkspaceLayout(a->B, a->H, a->n_slots).total;
}

int64_t kda_snapshot_count(const int32_t *cu, int32_t B, int32_t snap_interval) {
  if (B < 0 || snap_interval < 0 || (B > 0 && !cu)) return -1;
  if (snap_interval == 0) return 0;
  int64_t n = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t len = (int64_t)cu[b + 1] - cu[b];
    if (len < 0) return -1;
    n += len / snap_interval;
  }
  return n;
}

}  // extern "C"

namespace {

// The fused layer's arguments: host checks and the device-side view.
kda_status check_fused(const kda_fused_args *f, const kda_args *a, const void *xq, const void *xk,
                       const void *xv, kda::FusedParams *fp) {
  if (!f || !f->conv_w || !f->norm_w || !f->conv_pool) return KDA_ERR_INVALID_ARG;
  if (f->conv_width != kda::kConvW) return KDA_ERR_UNSUPPORTED;
  if (f->conv_act != 0 && f->conv_act != 1) return KDA_ERR_INVALID_ARG;
  if (!(f->norm_eps >= 0.f)) return KDA_ERR_INVALID_ARG;
  if (2 * a->dk + a->dv > 384) return KDA_ERR_UNSUPPORTED;
  if (a->T_total > 0) {
    const void *ps[] = {xq, xk, xv, f->gate};
    for (const void *p : ps)
      if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  }
  fp->xq = xq; fp->xk = xk; fp->xv = xv; fp->gate = f->gate;
  fp->conv_w = f->conv_w; fp->norm_w = f->norm_w; fp->conv_pool = f->conv_pool;
  fp->act = f->conv_act; fp->eps = f->norm_eps;
  return KDA_OK;
}

size_t elem_size(int32_t dtype) { return dtype == KDA_BF16 ? 2 : 4; }

// Scratch of the fused prefill: q, k, v (convolved) and o, each 256-byte aligned.
struct FusedScratch {
  size_t q, k, v, o, total;
  FusedScratch(const kda_args *a) {
    const size_t es = elem_size(a->dtype), T = (size_t)(a->T_total > 0 ? a->T_total : 0);
    const size_t nk = T * a->H * a->dk * es, nv = T * a->H * a->dv * es;
    q = 0;
    k = kda::align256(nk);
    v = k + kda::align256(nk);
    o = v + kda::align256(nv);
    total = o + kda::align256(nv);
  }
};

// Every prefill entry point: snapshots go to the dense buffer snaps, or, with
// a retention map snap_slots, into the pool slots it names (exactly one of the
// two is non-NULL when the call takes snapshots).  With fused (not NULL), q,
// k, v are the raw inputs, which the convolution turns into scratch; the
// recurrence writes its outputs into scratch and the gated RMSNorm into out.
kda_status prefill(const void *q, const void *k, const void *v, const void *g, const void *beta,
                   const int32_t *cu_seqlens, const int32_t *init_slots, float *state_pool,
                   void *out, int32_t snap_interval, float *snaps, const int32_t *snap_slots,
                   const kda_args *a, const kda_fused_args *fused = nullptr,
                   void *scratch = nullptr, size_t scratch_bytes = 0) {
  g_last_launches = 0;
  kda_status st = check_common(a);
  if (st != KDA_OK) return st;
  // the snapshot target may be NULL with an interval only when its capacity
  // is 0 (a batch whose sequences are all shorter than the interval)
  const bool target = snaps || snap_slots;
  if (snap_interval < 0 || a->snaps_capacity < 0) return KDA_ERR_INVALID_ARG;
  if (snaps && snap_slots) return KDA_ERR_INVALID_ARG;
  if (snap_interval == 0 && target) return KDA_ERR_INVALID_ARG;
  if (snap_interval > 0 && !target && a->snaps_capacity > 0) return KDA_ERR_INVALID_ARG;
  if (snaps && !aligned16(snaps)) return KDA_ERR_INVALID_ARG;
  if (a->algo < KDA_ALGO_AUTO || a->algo > KDA_ALGO_CHUNKED_COOP_HALVES) return KDA_ERR_INVALID_ARG;
  if (a->B == 0) return a->T_total == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
  if (!cu_seqlens || !init_slots || !state_pool || !aligned16(state_pool))
    return KDA_ERR_INVALID_ARG;
  if ((st = check_tokens(q, k, v, g, beta, out, a->T_total)) != KDA_OK) return st;
  kda::FusedParams fp;
  std::memset(&fp, 0, sizeof(fp));
  void *o_final = out;
  if (fused) {
    if ((st = check_fused(fused, a, q, k, v, &fp)) != KDA_OK) return st;
    const FusedScratch sc(a);
    if (!scratch || !aligned16(scratch) || scratch_bytes < sc.total) return KDA_ERR_INVALID_ARG;
    char *b = static_cast<char *>(scratch);
    q = b + sc.q;
    k = b + sc.k;
    v = b + sc.v;
    out = b + sc.o;
  }

  const kda::WorkspaceLayout lay(a->B, a->H, a->n_slots);
  char *ws = static_cast<char *>(a->workspace);
  kda::PrefillPlan p;
  std::memset(&p, 0, sizeof(p));
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.cu_seqlens = cu_seqlens; p.init_slots = init_slots;
  p.pool = state_pool; p.out = out; p.snaps = snaps; p.snap_slots = snap_slots;
  p.snap_interval = snap_interval;
  p.snaps_capacity = target ? a->snaps_capacity : 0;
  p.B = a->B; p.T_total = a->T_total; p.H = a->H; p.dk = a->dk; p.dv = a->dv;
  p.n_slots = a->n_slots; p.dtype = a->dtype;
  p.err = reinterpret_cast<uint32_t *>(ws);
  p.meta = reinterpret_cast<kda::SeqMeta *>(ws + lay.meta_off);
  p.order = reinterpret_cast<int32_t *>(ws + lay.order_off);
  p.claims = reinterpret_cast<uint32_t *>(ws + lay.claims_off);
  p.rerun = reinterpret_cast<uint32_t *>(ws + lay.rerun_off);
  if ((st = from_cuda(next_epoch(a, &p.epoch))) != KDA_OK) return st;
  p.stream = static_cast<cudaStream_t>(a->stream);
  if (lay.coop_units > 0) {
    p.coop_hdr = reinterpret_cast<uint32_t *>(ws + lay.coop_off);
    p.coop_flags = reinterpret_cast<unsigned long long *>(ws + lay.coop_flags_off);
    p.coop_ring = reinterpret_cast<uint8_t *>(ws + lay.coop_ring_off);
  }

  bool chunked = kda::chunked_supported(p);
  int mode = kda::kChunkAuto;
  if (a->algo == KDA_ALGO_CHUNKED_PER_STATE) mode = kda::kChunkPerState;
  if (a->algo == KDA_ALGO_CHUNKED_COOP) {
    if (!kda::coop_supported(p)) return KDA_ERR_UNSUPPORTED;
    mode = kda::kChunkCoop;
  }
  if (a->algo == KDA_ALGO_CHUNKED_COOP_HALVES) {
    if (!kda::coop_halves_supported(p)) return KDA_ERR_UNSUPPORTED;
    mode = kda::kChunkCoopHalves;
  }
  if (a->algo >= KDA_ALGO_CHUNKED && !chunked) return KDA_ERR_UNSUPPORTED;
  if (a->algo == KDA_ALGO_RECURRENT) chunked = false;

  if ((st = from_cuda(kda::launch_meta(p))) != KDA_OK) return st;
  g_last_launches = 1;
  if (fused) {  // the convolution, then the new convolution states
    if ((st = from_cuda(kda::launch_conv_prefill(p, fp))) != KDA_OK) return st;
    if ((st = from_cuda(kda::launch_conv_state(p, fp))) != KDA_OK) return st;
    g_last_launches += 2;
  }
  record(a->ev_begin, p.stream);
  st = from_cuda(chunked ? kda::launch_chunked_prefill(p, mode) : kda::launch_recurrent_prefill(p));
  record(a->ev_end, p.stream);
  if (st != KDA_OK) return st;
  ++g_last_launches;
  if (chunked) {
    // units whose decay left the chunked algorithm's exponent range are
    // recomputed by the exact token-recurrent kernel (every other CTA of this
    // launch returns at once)
    if ((st = from_cuda(kda::launch_recurrent_prefill(p, true))) != KDA_OK) return st;
    ++g_last_launches;
  }
  if (fused) {  // the gated RMSNorm of the recurrence's outputs
    if ((st = from_cuda(kda::launch_rms_gate(p, fp, out, o_final))) != KDA_OK) return st;
    ++g_last_launches;
  }
  return st;
}

}  // namespace

extern "C" {

kda_status kda_prefill_varlen(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, const int32_t *cu_seqlens,
                              const int32_t *init_slots, float *state_pool, void *out,
                              int32_t snap_interval, float *snaps, const kda_args *a) {
  return prefill(q, k, v, g, beta, cu_seqlens, init_slots, state_pool, out, snap_interval, snaps,
                 nullptr, a);
}

kda_status kda_prefill_varlen_retain(const void *q, const void *k, const void *v, const void *g,
                                     const void *beta, const int32_t *cu_seqlens,
                                     const int32_t *init_slots, float *state_pool, void *out,
                                     int32_t snap_interval, const int32_t *snap_slots,
                                     const kda_args *a) {
  return prefill(q, k, v, g, beta, cu_seqlens, init_slots, state_pool, out, snap_interval,
                 nullptr, snap_slots, a);
}

kda_status kda_prefill_varlen_fused(const void *xq, const void *xk, const void *xv,
                                    const void *g, const void *beta, const int32_t *cu_seqlens,
                                    const int32_t *init_slots, float *state_pool, void *out,
                                    int32_t snap_interval, float *snaps, const kda_fused_args *f,
                                    void *scratch, size_t scratch_bytes, const kda_args *a) {
  if (!f) {
    g_last_launches = 0;
    return KDA_ERR_INVALID_ARG;
  }
  return prefill(xq, xk, xv, g, beta, cu_seqlens, init_slots, state_pool, out, snap_interval,
                 snaps, nullptr, a, f, scratch, scratch_bytes);
}

size_t kda_fused_scratch_bytes(const kda_args *a) {
  if (!a || a->T_total < 0 || a->H <= 0 || a->dk <= 0 || a->dv <= 0) return 0;
  return FusedScratch(a).total;
}

kda_status kda_decode_fused(const void *xq, const void *xk, const void *xv, const void *g,
                            const void *beta, const int32_t *slot_ids, float *state_pool,
                            void *out, int32_t n_tok, float *per_tok_states,
                            const kda_fused_args *f, const kda_args *a) {
  g_last_launches = 0;
  kda_status st = check_common(a);
  if (st != KDA_OK) return st;
  if (a->dk != 128 || a->dv != 128) return KDA_ERR_UNSUPPORTED;
  if (n_tok < 1 || (int64_t)a->B * n_tok != a->T_total) return KDA_ERR_INVALID_ARG;
  if (a->B == 0) return KDA_OK;
  if (!slot_ids || !state_pool || !aligned16(state_pool)) return KDA_ERR_INVALID_ARG;
  if (per_tok_states && !aligned16(per_tok_states)) return KDA_ERR_INVALID_ARG;
  if ((st = check_tokens(xq, xk, xv, g, beta, out, a->T_total)) != KDA_OK) return st;
  kda::FusedParams fp;
  if ((st = check_fused(f, a, xq, xk, xv, &fp)) != KDA_OK) return st;

  const kda::WorkspaceLayout lay(a->B, a->H, a->n_slots);
  char *ws = static_cast<char *>(a->workspace);
  kda::DecodePlan p;
  std::memset(&p, 0, sizeof(p));
  p.g = g; p.beta = beta;
  p.slot_ids = slot_ids; p.pool = state_pool; p.out = out; p.per_tok = per_tok_states;
  p.N = a->B; p.n_tok = n_tok; p.H = a->H; p.dk = a->dk; p.dv = a->dv;
  p.n_slots = a->n_slots; p.dtype = a->dtype;
  p.err = reinterpret_cast<uint32_t *>(ws);
  p.claims = reinterpret_cast<uint32_t *>(ws + lay.claims_off);
  if ((st = from_cuda(next_epoch(a, &p.epoch))) != KDA_OK) return st;
  p.stream = static_cast<cudaStream_t>(a->stream);
  record(a->ev_begin, p.stream);
  st = from_cuda(kda::launch_decode_fused(p, fp));
  record(a->ev_end, p.stream);
  if (st == KDA_OK) g_last_launches = 1;
  return st;
}

kda_status kda_decode(const void *q, const void *k, const void *v, const void *g,
                      const void *beta, const int32_t *slot_ids, float *state_pool, void *out,
                      int32_t n_tok, float *per_tok_states, const kda_args *a) {
  g_last_launches = 0;
  kda_status st = check_common(a);
  if (st != KDA_OK) return st;
  if (n_tok < 1 || (int64_t)a->B * n_tok != a->T_total) return KDA_ERR_INVALID_ARG;
  if (a->B == 0) return KDA_OK;
  if (!slot_ids || !state_pool || !aligned16(state_pool)) return KDA_ERR_INVALID_ARG;
  if (per_tok_states && !aligned16(per_tok_states)) return KDA_ERR_INVALID_ARG;
  if ((st = check_tokens(q, k, v, g, beta, out, a->T_total)) != KDA_OK) return st;

  const kda::WorkspaceLayout lay(a->B, a->H, a->n_slots);
  char *ws = static_cast<char *>(a->workspace);
  kda::DecodePlan p;
  std::memset(&p, 0, sizeof(p));
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.slot_ids = slot_ids; p.pool = state_pool; p.out = out; p.per_tok = per_tok_states;
  p.N = a->B; p.n_tok = n_tok; p.H = a->H; p.dk = a->dk; p.dv = a->dv;
  p.n_slots = a->n_slots; p.dtype = a->dtype;
  p.err = reinterpret_cast<uint32_t *>(ws);
  p.claims = reinterpret_cast<uint32_t *>(ws + lay.claims_off);
  if ((st = from_cuda(next_epoch(a, &p.epoch))) != KDA_OK) return st;
  p.stream = static_cast<cudaStream_t>(a->stream);
  const bool fast = a->dk == 128 && a->dv == 128;
  record(a->ev_begin, p.stream);
  st = from_cuda(fast ? kda::launch_decode128(p) : kda::launch_recurrent_decode(p));
  record(a->ev_end, p.stream);
  if (st == KDA_OK) g_last_launches = 1;
  return st;
}

kda_status kda_decode_spec(const void *q, const void *k, const void *v, const void *g,
                           const void *beta, const int32_t *slot_ids, float *state_pool,
                           void *out, int32_t n_tok, const void *k_prev, const void *v_prev,
                           const void *g_prev, const void *beta_prev,
                           const int32_t *accepted_prev, int32_t n_prev, const kda_args *a) {
  g_last_launches = 0;
  kda_status st = check_common(a);
  if (st != KDA_OK) return st;
  if (n_tok < 0 || n_prev < 0 || (int64_t)a->B * n_tok != a->T_total) return KDA_ERR_INVALID_ARG;
  if (a->B == 0) return KDA_OK;
  if (!slot_ids || !state_pool || !aligned16(state_pool)) return KDA_ERR_INVALID_ARG;
  if ((st = check_tokens(q, k, v, g, beta, out, a->T_total)) != KDA_OK) return st;
  if (n_prev > 0) {
    const void *ps[] = {k_prev, v_prev, g_prev, beta_prev};
    for (const void *p : ps)
      if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (!accepted_prev) return KDA_ERR_INVALID_ARG;
  }

  const kda::WorkspaceLayout lay(a->B, a->H, a->n_slots);
  char *ws = static_cast<char *>(a->workspace);
  kda::DecodePlan p;
  std::memset(&p, 0, sizeof(p));
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.slot_ids = slot_ids; p.pool = state_pool; p.out = out; p.per_tok = nullptr;
  p.N = a->B; p.n_tok = n_tok; p.H = a->H; p.dk = a->dk; p.dv = a->dv;
  p.n_slots = a->n_slots; p.dtype = a->dtype;
  p.err = reinterpret_cast<uint32_t *>(ws);
  p.claims = reinterpret_cast<uint32_t *>(ws + lay.claims_off);
  if ((st = from_cuda(next_epoch(a, &p.epoch))) != KDA_OK) return st;
  p.stream = static_cast<cudaStream_t>(a->stream);
  p.spec = 1;
  p.n_prev = n_prev;
  p.k_prev = k_prev; p.v_prev = v_prev; p.g_prev = g_prev; p.beta_prev = beta_prev;
  p.accepted = accepted_prev;
  const bool fast = a->dk == 128 && a->dv == 128;
  record(a->ev_begin, p.stream);
  st = from_cuda(fast ? kda::launch_decode128(p) : kda::launch_recurrent_decode(p));
  record(a->ev_end, p.stream);
  if (st == KDA_OK) g_last_launches = 1;
  return st;
}

kda_status kda_device_status(const kda_args *a, uint32_t *detail) {
  if (detail) *detail = 0;
  if (!a || !a->workspace) return KDA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(a->stream);
  uint32_t bits = 0;
  if (cudaMemcpyAsync(&bits, a->workspace, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
  if (bits) {
    if (cudaMemsetAsync(a->workspace, 0, sizeof(bits), s) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
  }
  if (detail) *detail = bits;
  if (bits & kda::ERR_TIMEOUT) return KDA_ERR_TIMEOUT;
  return bits ? KDA_ERR_DEVICE_CHECK : KDA_OK;
}

const char *kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_DEVICE_CHECK: return "KDA_ERR_DEVICE_CHECK";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
  }
  return "KDA_ERR_UNKNOWN";
}

int32_t kda_last_launch_count(void) { return g_last_launches; }

}  // extern "C"
