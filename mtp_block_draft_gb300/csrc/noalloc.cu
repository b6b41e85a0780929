// dmtp_t1_head_noalloc: the first-candidate head (RMSNorm, LM head, row argmax) for
// callers that must not allocate device memory.
//
// Some embedders cannot call cudaMalloc: a serving engine that owns a fixed memory pool
// and forbids allocations outside it, or a latency-critical path where cudaMalloc /
// cudaFree would synchronise the device. The round library already takes all of its
// memory from the caller; this entry point goes further and needs no workspace at all.
// Its scratch - the bf16 operand of the head GEMM and the packed argmax keys - is
// a file-scope __device__ array of fixed size that every GPU loading the library holds
// until the process exits.
//
// The array holds 32 x 4096 bf16 operand elements and 32 eight-byte keys: 262,400 bytes
// (about 0.26 MB) per GPU.
//
// The first call on a device sets up that device (it looks up the array's device address
// with cudaGetSymbolAddress and raises the head kernel's shared-memory limit); make that
// first call before any stream capture. The set-up is kept per device index for the life
// of the process and does not survive cudaDeviceReset (the context it was made in is
// gone): a caller that resets a device must not call this entry point on it afterwards.
// All calls share the one array: calls that may overlap on the GPU (other streams, other
// threads) race on it and must be serialised by the caller.
#include <mutex>

#include "../../include/dmtp.h"
#include "common.cuh"
#include "ops.h"

namespace {

constexpr int kMaxRows = DMTP_NOALLOC_MAX_ROWS;  // token rows per call
constexpr int kMaxD = DMTP_NOALLOC_MAX_DMODEL;   // hidden size
constexpr size_t kOperandBytes = (size_t)kMaxRows * kMaxD * 2;  // rows x d, bf16
constexpr size_t kKeyBytes = (size_t)kMaxRows * 8;

// The scratch: the GEMM operand, then the argmax keys.
static __device__ __align__(256) unsigned char g_scratch[kOperandBytes + kKeyBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
int g_nsm[kMaxDevices] = {};

int device_scratch(void** out, int* nsm) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DMTP_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return DMTP_ECUDA;
    if (dmtp::head_init_attributes()) return DMTP_ECUDA;
    if (cudaDeviceGetAttribute(&g_nsm[dev], cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return DMTP_ECUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  *nsm = g_nsm[dev];
  return DMTP_OK;
}

}  // namespace

extern "C" int dmtp_t1_head_noalloc(const void* head, const void* norm_gain, const float* h,
                                    int rows, int vocab, int d_model, float eps, int32_t* ids,
                                    float* logits, void* stream) {
  if (!head || !norm_gain || !h || !ids) return DMTP_EINVAL;
  if (rows < 1 || rows > kMaxRows || d_model < 64 || d_model > kMaxD || d_model % 64 ||
      vocab < 1 || ((uintptr_t)head & 15))
    return DMTP_EINVAL;
  // an error left pending by earlier work on this thread is reported, not cleared, and
  // nothing is launched
  if (cudaPeekAtLastError() != cudaSuccess) return DMTP_ECUDA;
  void* base = nullptr;
  int nsm = 0;
  int r = device_scratch(&base, &nsm);
  if (r) return r;
  cudaStream_t st = (cudaStream_t)stream;
  void* X = base;
  unsigned long long* keys = (unsigned long long*)((char*)base + kOperandBytes);
  dmtp::HeadPlan plan;
  // the round's LM-head kernel on the same single-bf16 operand; the shapes were checked
  // above, so a failure here is the tensor-map encoding
  if (dmtp::head_plan(&plan, head, vocab, d_model, X, rows, nsm, 256, 8)) return DMTP_ECUDA;
  // keys start at zero for the atomic max; the operand rows are fully rewritten
  if (cudaMemsetAsync(keys, 0, (size_t)rows * 8, st) != cudaSuccess) return DMTP_ECUDA;
  dmtp::pdl_fence();  // the next launch follows a memset: no programmatic overlap
  dmtp::op_rmsnorm(1, h, d_model, norm_gain, X, d_model, 0, nullptr, 0,
                   nullptr, 0, 0, rows, d_model, eps, dmtp::RowMap(), st);
  dmtp::op_head_tc(plan, keys, logits, vocab, nullptr, nullptr, st);
  dmtp::op_keys_to_ids(keys, rows, 1, ids, 1, 0, nullptr, 0, 0, st);
  // no error was pending on entry, so one now comes from these launches (consumed here)
  return cudaGetLastError() == cudaSuccess ? DMTP_OK : DMTP_ECUDA;
}
