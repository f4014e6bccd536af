// Step composer: the layer calls a prompt's prefill is cut into by the serving loop of the
// "moe-prefill-quantum" page (host code only; see include/moe.h for the contract).
//
// Two levels.  The server hands the prompt to the engine in pieces counted from the prompt's
// first token: `quantum` tokens while any request is generating, 2048 otherwise (the cause
// section's source excerpt).  The engine runs a piece as one or more calls, ending a call at the
// next multiple of prefill_cap in absolute context position (the prefill_cap section's excerpt),
// so a prompt that starts off a boundary is cut 2048, 509, 1539, ... and never realigns.  A call
// is at most prefill_cap tokens (the engine's batch buffer), so pieces above prefill_cap are cut
// at the boundaries too.
#include <cstdint>

#include "kernels.h"

namespace {

constexpr int32_t kIdlePiece = 2048;  // piece size while nothing is generating

}  // namespace

extern "C" moe_status moe_compose_prefill(int64_t start_pos, int64_t n_tokens, int32_t quantum,
                                          int32_t generation_active, int32_t prefill_cap,
                                          moe_prefill_call* calls, int64_t max_calls, int64_t* n_calls) {
  if (!n_calls) return moe::fail_message(MOE_ERR_INVALID_ARG, "n_calls is required");
  if (start_pos < 0 || n_tokens < 0 || quantum < 1 || prefill_cap < 1)
    return moe::fail_message(MOE_ERR_INVALID_ARG, "need start_pos >= 0, n_tokens >= 0, quantum >= 1, prefill_cap >= 1");
  if (max_calls < 0 || (max_calls > 0 && !calls))
    return moe::fail_message(MOE_ERR_INVALID_ARG, "calls is required when max_calls > 0");
  const int64_t piece = generation_active ? quantum : kIdlePiece;
  const int64_t cap = prefill_cap;
  int64_t count = 0, pos = start_pos, done = 0;
  int32_t piece_index = 0;
  while (done < n_tokens) {
    const int64_t piece_end = done + (piece < n_tokens - done ? piece : n_tokens - done);
    while (done < piece_end) {
      int64_t n = piece_end - done;
      if (n > cap) n = cap;
      const int64_t to_boundary = cap - pos % cap;  // == cap on a boundary
      if (n > to_boundary) n = to_boundary;
      if (count < max_calls) calls[count] = moe_prefill_call{pos, static_cast<int32_t>(n), piece_index};
      ++count;
      pos += n;
      done += n;
    }
    ++piece_index;
  }
  *n_calls = count;
  return MOE_OK;
}
