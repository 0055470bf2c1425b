// Routing for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc and have no spare buffer to lend as a
// workspace: a host runtime that owns every byte of device memory through its own arena and
// forbids third-party code from allocating (so that its accounting stays exact and no
// allocation stalls the device in the middle of a step), or a plugin interface that hands the
// library only its input and output tensors.  moe_route_topk_noalloc serves them: its scratch
// space (the per-block expert histograms and their prefix sums) is a fixed array inside the
// library, so a call needs nothing beyond its inputs and outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "moe_gb300.h"

namespace moe {

// The expert histogram: ceil(T / 128) rows of route_ldh(E) bytes (E rounded up to a power of two
// of at least 16), 128 KB at most -- the size the slots kernel reads whole, so these calls never
// need the larger histograms' row-prefix table.  Every GPU that loads the library holds this
// array until the process exits.
constexpr int NOALLOC_ROUTE_MAX_BYTES = static_cast<int>(ROUTE_DIRECT_BYTES);
static __device__ __align__(256) uint8_t g_route_scratch[NOALLOC_ROUTE_MAX_BYTES];

static SymbolCache g_scratch_sym;

// Device address of the array in the current device's context: looked up (cudaGetSymbolAddress)
// on the first call on a device, and again whenever the device's context has changed since (a
// cudaDeviceReset in between), so the kernels never receive a stale address.
static int route_scratch(uint8_t** out) {
  void* p = nullptr;
  MOE_TRY(symbol_address(g_route_scratch, &g_scratch_sym, &p, "moe_route_topk_noalloc"));
  *out = static_cast<uint8_t*>(p);
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_route_topk_noalloc(const moe_cfg* c, const void* x, const void* W_r,
                                      const float* b_r, const float* logits_in, float* logits_out,
                                      int32_t* idx, float* gate, int32_t* counts, int32_t* offsets,
                                      int32_t* slot_of_pair, int32_t* token_of_slot,
                                      void* stream) {
  MOE_TRY(validate_cfg(c));
  if (!logits_in && !logits_out) {
    set_error("moe_route_topk_noalloc: logits_in or logits_out must be given (the router "
              "logits need a caller buffer)");
    return MOE_ERR_INVALID_ARG;
  }
  const int64_t bytes = route_hist_bytes(c->T, c->E);
  if (bytes > NOALLOC_ROUTE_MAX_BYTES) {
    set_error("moe_route_topk_noalloc: ceil(T/128) * E16 = %lld (E16: E rounded up to a power "
              "of two, at least 16) exceeds the built-in scratch of %d bytes (e.g. T=65536 with "
              "E=256); use moe_route_topk with a workspace",
              static_cast<long long>(bytes), NOALLOC_ROUTE_MAX_BYTES);
    return MOE_ERR_UNSUPPORTED;
  }
  MOE_TRY(validate_ptr(x, "x", !logits_in));
  MOE_TRY(validate_ptr(W_r, "W_r", !logits_in));
  MOE_TRY(validate_ptr(b_r, "b_r", false));
  MOE_TRY(validate_ptr(logits_in, "logits_in", false));
  MOE_TRY(validate_ptr(logits_out, "logits_out", false));
  MOE_TRY(validate_ptr(idx, "idx", true));
  MOE_TRY(validate_ptr(gate, "gate", true));
  MOE_TRY(validate_ptr(counts, "counts", true));
  MOE_TRY(validate_ptr(offsets, "offsets", true));
  MOE_TRY(validate_ptr(slot_of_pair, "slot_of_pair", true));
  MOE_TRY(validate_ptr(token_of_slot, "token_of_slot", true));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * c->E, st) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c->E + 1), st) != cudaSuccess) {
      set_error("moe_route_topk_noalloc: cudaMemsetAsync failed");
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  uint8_t* hist = nullptr;
  MOE_TRY(route_scratch(&hist));
  // every histogram row is written in full (by the top-k kernel or the router GEMM) before the
  // slots kernel reads it, so the array needs no clearing between calls
  return route_stages(c, x, W_r, b_r, logits_in, logits_out, idx, gate, counts, offsets,
                      slot_of_pair, token_of_slot, hist, nullptr, st);
}
