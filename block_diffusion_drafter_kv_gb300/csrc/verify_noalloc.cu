// Greedy verification for callers that cannot allocate device memory.
//
// dflash_verify_greedy needs a few hundred kilobytes of scratch (per-chunk argmax
// partials and per-sequence arrival counters), which normally live in the workspace the
// caller allocates and binds to a handle. Some callers cannot allocate at all: code that
// runs inside another engine's decode loop on a memory pool that forbids new
// allocations, or a host process that is only handed logits and token buffers. For them
// this file keeps that scratch in one fixed array compiled into the library, and the
// entry point below takes no handle and allocates nothing.
#include <algorithm>
#include <mutex>

#include "dflash.h"
#include "internal.h"

namespace {

constexpr int kChunks = DFLASH_NOALLOC_MAX_CHUNKS;
constexpr int kMaxBatch = DFLASH_NOALLOC_MAX_BATCH;
constexpr int kMaxBlock = 16;

// Layout of the array, in 4-byte words:
//   [0, 64)                          error flag and padding
//   [64, 64 + kMaxBatch)             per-sequence arrival counters (must start at zero)
//   then part_v, part_i              [kMaxBatch][kMaxBlock][kChunks] each
constexpr size_t kCntOff = 64;
constexpr size_t kPartVOff = kCntOff + kMaxBatch;
constexpr size_t kPartIOff = kPartVOff + static_cast<size_t>(kMaxBatch) * kMaxBlock * kChunks;
constexpr size_t kWords = kPartIOff + static_cast<size_t>(kMaxBatch) * kMaxBlock * kChunks;

// Every GPU that loads the library holds this array (about 257 KB) until the process exits.
static __device__ __align__(256) int g_verify_scratch[kWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_verify_scratch on the current device, looked up once per device.
// The name itself is only a host-side stand-in for the symbol and must never be passed
// to a kernel.
int* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return nullptr;
    g_scratch_ptr[dev] = static_cast<int*>(p);
  }
  return g_scratch_ptr[dev];
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

}  // namespace

extern "C" int dflash_verify_greedy_noalloc(const float* target_logits, const int32_t* drafted, int32_t batch,
                                            int32_t block, int32_t vocab, int32_t* accept_len,
                                            int32_t* committed, int32_t* last_token, void* stream) {
  if (!target_logits || !accept_len || !committed || !last_token || (block > 1 && !drafted)) return DFLASH_E_INVAL;
  if (batch < 1 || block < 1 || vocab < 2 || vocab > DFLASH_NOALLOC_MAX_VOCAB) return DFLASH_E_INVAL;
  // the logits are read 16 bytes at a time, the token arrays as 4-byte words
  auto misaligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (misaligned(target_logits, 16) || misaligned(drafted, 4) || misaligned(accept_len, 4) ||
      misaligned(committed, 4) || misaligned(last_token, 4))
    return DFLASH_E_INVAL;
  if (batch > kMaxBatch || block > kMaxBlock) return DFLASH_E_CAPACITY;
  int* scratch = scratch_for_current_device();
  if (!scratch) return DFLASH_E_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The arrival counters must start every call at zero; the kernel also leaves them at
  // zero, but a call that failed part-way could not have.
  if (cudaMemsetAsync(scratch + kCntOff, 0, sizeof(int) * kMaxBatch, st) != cudaSuccess) return DFLASH_E_CUDA;
  dfl::VerifyParams P{};
  P.logits = target_logits;
  P.drafted = drafted;
  P.accept_len = accept_len;
  P.committed = committed;
  P.last_token = last_token;
  P.err = scratch;
  P.seq_cnt = scratch + kCntOff;
  P.part_v = reinterpret_cast<float*>(scratch + kPartVOff);
  P.part_i = scratch + kPartIOff;
  P.B = block;
  P.V = vocab;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DFLASH_E_CUDA;
  const int chunks = std::max(1, std::min(kChunks, ceil_div(2LL * sms, static_cast<long long>(batch) * block)));
  P.chunk_len = ceil_div(ceil_div(vocab, chunks), 1024) * 1024;
  P.chunks = ceil_div(vocab, P.chunk_len);
  return dfl::launch_verify(P, batch, st, false) == 0 ? DFLASH_OK : DFLASH_E_CUDA;
}
