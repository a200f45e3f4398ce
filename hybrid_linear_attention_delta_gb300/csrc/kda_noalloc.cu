// kda_noalloc.cu -- kda_decode_noalloc: the dk = dv = 128 decode step for
// callers that cannot hand the library a workspace.
//
// Who needs this: code that runs inside a host framework which owns all device
// memory through its own pool (a serving engine's state-cache manager, a
// plugin that is given only the step's tensors) or that sits on a latency
// path where cudaMalloc is not allowed, because it may synchronise the whole
// device.  Such callers can pass inputs and outputs but cannot allocate the
// workspace that kda_decode needs for its duplicate-slot claims.
//
// This variant launches the same decode kernel with its scratch taken from a
// file-scope device array instead.  The array is part of the library image:
// every GPU that loads libkda.so holds it (kNoallocScratchBytes, 2 MiB + 256 B)
// until the process exits.  Its device address is looked up once per device
// with cudaGetSymbolAddress; the host symbol itself is only a stand-in and is
// never given to a kernel.
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

// Largest n_slots * H the shared claim table covers.
constexpr int64_t kNoallocMaxStates = 131072;
constexpr size_t kNoallocScratchWords = 64 + (size_t)kNoallocMaxStates * kClaimsPerState;

// word 0: error bits of calls that pass no err_bits pointer (a sink, never
// read); words 64..: claim stamps, one group of kClaimsPerState per state.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoallocScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
uint32_t *g_scratch_ptr[kMaxDevices] = {};
// per device: the epoch of the last call, the stamp its claims carry
uint32_t g_epoch[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call per device) and the epoch of this call there; *wrapped is set
// when that device's 32-bit epoch count has just wrapped, so that every stamp
// left in its table could equal a new epoch.  nullptr when the lookup fails.
uint32_t *scratch_on_current_device(uint32_t *epoch, bool *wrapped) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = static_cast<uint32_t *>(ptr);
  }
  *wrapped = ++g_epoch[dev] == 0;  // 0 marks "never claimed"
  if (*wrapped) g_epoch[dev] = 1;
  *epoch = g_epoch[dev];
  return g_scratch_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kda

extern "C" kda_status kda_decode_noalloc(const void *q, const void *k, const void *v,
                                         const void *g, const void *beta,
                                         const int32_t *slot_ids, float *state_pool, void *out,
                                         int32_t n_tok, float *per_tok_states, uint32_t *err_bits,
                                         const kda_args *a) {
  using namespace kda;
  if (!a || (a->dtype != KDA_F32 && a->dtype != KDA_BF16)) return KDA_ERR_INVALID_ARG;
  if (a->dk != 128 || a->dv != 128) return KDA_ERR_UNSUPPORTED;
  if (a->B < 0 || a->H <= 0 || a->n_slots <= 0 || n_tok < 1 ||
      (int64_t)a->B * n_tok != a->T_total)
    return KDA_ERR_INVALID_ARG;
  if ((int64_t)a->n_slots * a->H > kNoallocMaxStates) return KDA_ERR_INVALID_ARG;
  if (a->B == 0) return KDA_OK;
  const void *ps[] = {q, k, v, g, beta, out, state_pool};
  for (const void *p : ps)
    if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
  if (!slot_ids || (per_tok_states && !aligned16(per_tok_states))) return KDA_ERR_INVALID_ARG;

  uint32_t epoch = 0;
  bool wrapped = false;
  uint32_t *scratch = scratch_on_current_device(&epoch, &wrapped);
  if (!scratch) return KDA_ERR_CUDA;
  // after 2^32 - 1 calls on a device the claim table is cleared once, on the
  // call's stream (a memset of the library's own array: nothing is allocated)
  if (wrapped && cudaMemsetAsync(scratch, 0, kNoallocScratchWords * sizeof(uint32_t),
                                 static_cast<cudaStream_t>(a->stream)) != cudaSuccess)
    return KDA_ERR_CUDA;

  DecodePlan p = {};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.slot_ids = slot_ids; p.pool = state_pool; p.out = out; p.per_tok = per_tok_states;
  p.N = a->B; p.n_tok = n_tok; p.H = a->H; p.dk = a->dk; p.dv = a->dv;
  p.n_slots = a->n_slots; p.dtype = a->dtype;
  p.err = err_bits ? err_bits : scratch;
  p.claims = scratch + 64;
  p.epoch = epoch;
  p.stream = static_cast<cudaStream_t>(a->stream);
  return launch_decode128(p) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
