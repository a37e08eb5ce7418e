// vfy_accept_static: the fused argmax + acceptance of vfy_accept for callers that cannot allocate
// device memory. Some callers cannot call cudaMalloc at all: code that runs inside a memory pool
// or allocator it must not re-enter, plug-ins whose host process owns every device allocation,
// and setups that have fixed their whole memory budget before decoding starts. vfy_accept needs a
// context (created with vfy_create, which allocates its workspace); this entry point needs none.
// Its scratch (per-row argmax keys, the CTA ticket, an error word) is a fixed array in this
// library's device memory, which every GPU that loads the library holds until the process exits.
#include <mutex>

#include "ptx.cuh"
#include "vfy_internal.cuh"

namespace vfy {
namespace {

constexpr int kStaticMaxRows = 1024;   // logit rows per call (sum over sequences of D_b + 1)
constexpr int kMaxDevices = 64;

// [0, kStaticMaxRows): argmax keys; [kStaticMaxRows]: ticket (low 32 bits); [kStaticMaxRows + 1]:
// error word (low 32 bits). 8 KiB + 16 bytes.
static __device__ __align__(256) unsigned long long g_accept_scratch[kStaticMaxRows + 2];

struct DeviceState {
  unsigned long long* scratch = nullptr;   // device address of g_accept_scratch on this device
  CUcontext ctx = nullptr;                 // the context that address belongs to
  int num_sms = 0;
};
std::mutex g_lock;
DeviceState g_state[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's current context, through the runtime's entry-point query (no link to libcuda).
bool current_context(CUcontext* out) {
  static CtxGetCurrentFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<CtxGetCurrentFn>(p);
  }
  return fn(out) == CUDA_SUCCESS;
}

// With the device current: look up the device address of the scratch array. (In host code,
// g_accept_scratch names a host-side stand-in, not device memory.) The address is cached per
// device and looked up again when the device's context has changed (after cudaDeviceReset the
// old address is gone).
cudaError_t device_state(int dev, DeviceState* out) {
  std::lock_guard<std::mutex> guard(g_lock);
  DeviceState& st = g_state[dev];
  CUcontext cur = nullptr;
  if (!current_context(&cur)) return cudaErrorUnknown;
  if (st.scratch == nullptr || st.ctx != cur) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_accept_scratch);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // cudaGetSymbolAddress made the device's primary context current if none was
    if (!current_context(&cur)) return cudaErrorUnknown;
    st.scratch = static_cast<unsigned long long*>(ptr);
    st.ctx = cur;
    st.num_sms = sms;
  }
  *out = st;
  return cudaSuccess;
}

}  // namespace
}  // namespace vfy

extern "C" vfy_status vfy_accept_static(const float* logits, int vocab, const int32_t* drafts,
                                        const int32_t* cu_rows, int num_seqs, int max_rows,
                                        int32_t* accepted_len, int32_t* bonus, int32_t* committed,
                                        int32_t* device_error, vfy_stream_t stream) {
  using namespace vfy;
  if (logits == nullptr || drafts == nullptr || cu_rows == nullptr || accepted_len == nullptr ||
      bonus == nullptr || committed == nullptr)
    return VFY_EINVAL;
  if (vocab < 1 || num_seqs < 1 || max_rows < num_seqs) return VFY_EINVAL;
  if (max_rows > kStaticMaxRows) return VFY_EINVAL;   // beyond the fixed scratch: refused
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0) return VFY_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    (void)cudaGetLastError();
    return VFY_ECUDA;
  }
  if (dev >= kMaxDevices) return VFY_EUNSUPPORTED;   // beyond the per-device address cache
  DeviceState st;
  if (device_state(dev, &st) != cudaSuccess) {
    (void)cudaGetLastError();
    return VFY_ECUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the last call's contents: start every call from zero keys, ticket and error.
  if (cudaMemsetAsync(st.scratch, 0, sizeof(unsigned long long) * (kStaticMaxRows + 2), s) != cudaSuccess) {
    (void)cudaGetLastError();
    return VFY_ECUDA;
  }
  AcceptParams p;
  p.logits = logits;
  p.vocab = vocab;
  p.drafts = drafts;
  p.cu_rows = cu_rows;
  p.num_seqs = num_seqs;
  p.max_rows = max_rows;
  int parts = static_cast<int>((2LL * st.num_sms + max_rows - 1) / max_rows);
  const int max_parts = (vocab + 1023) / 1024;
  if (parts > max_parts) parts = max_parts;
  if (parts < 1) parts = 1;
  int seg = (vocab + parts - 1) / parts;
  seg = (seg + 3) & ~3;
  p.parts = (vocab + seg - 1) / seg;
  p.seg = seg;
  p.accepted_len = accepted_len;
  p.bonus = bonus;
  p.committed = committed;
  p.keys = st.scratch;
  p.counter = reinterpret_cast<unsigned int*>(st.scratch + kStaticMaxRows);
  p.stable_metadata = 0;
  p.err = device_error != nullptr ? device_error : reinterpret_cast<int*>(st.scratch + kStaticMaxRows + 1);
  const bool vec4 = (vocab % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  if (launch_accept(p, vec4, s) != cudaSuccess) {
    (void)cudaGetLastError();
    return VFY_ECUDA;
  }
  return VFY_OK;
}
