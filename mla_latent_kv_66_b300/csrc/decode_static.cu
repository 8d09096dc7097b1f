// Allocation-free decode entry point: mla_decode + mla_split_kv_combine with
// their scratch workspace in a fixed-size array that lives in this library's
// device image, so the caller passes only inputs and outputs.
//
// Who needs it: code that is handed device buffers but may not create any,
// e.g. a plugin inside a host application or serving runtime that reserves
// all device memory in its own pool up front, or a latency-critical path
// where cudaMalloc (which can synchronise the device) is not acceptable.
#include <mutex>

#include "common.cuh"

namespace {

// Scratch for the error word, split records, sequence page offsets, the
// split-KV partial results and (8-bit tensor-core modes) the E4M3 query.  Every GPU that loads the library holds it until
// the process exits.  Every call shares it.
constexpr size_t kStaticWsBytes = 32u << 20;
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 64;
void* g_static_ptr[kMaxDevices];
std::mutex g_static_mu;

// Device address of g_static_ws on the current device.  In host code the
// array's name is only a host-side stand-in, so its address has to be asked
// for once per device, with that device current.
cudaError_t static_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return e;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" mla_status mla_decode_static(const mla_params* p, const void* q_lat, const void* q_pe,
                                        const void* ckv_cache, const void* kpe_cache,
                                        const float* kv_scale, const int32_t* page_table,
                                        const int32_t* seq_lens, void* o_lat, float* lse,
                                        mla_stream_t stream) {
  // largest worker count (at most the automatic one) whose workspace fits
  int G = mla_decode_num_splits(p, 0);
  if (G < 1) return MLA_ERR_INVALID_ARG;
  while (G >= 1 && mla_decode_workspace_size(p, G) > kStaticWsBytes) --G;
  if (G < 1) return MLA_ERR_WORKSPACE;  // B or H too large for the fixed scratch
  void* ws = nullptr;
  if (static_ws_address(&ws) != cudaSuccess) return MLA_ERR_CUDA;
  // the sticky error word must start at zero; everything else the kernels
  // read is written earlier in the same call
  if (cudaMemsetAsync(ws, 0, sizeof(int), (cudaStream_t)stream) != cudaSuccess) return MLA_ERR_CUDA;
  mla_status s = mla_decode(p, q_lat, q_pe, ckv_cache, kpe_cache, kv_scale, page_table, seq_lens, G,
                            ws, kStaticWsBytes, o_lat, lse, stream);
  if (s != MLA_OK) return s;
  return mla_split_kv_combine(p, ws, kStaticWsBytes, G, o_lat, lse, stream);
}

// The error word of the fixed scratch (offset 0, the same word mla_decode
// keeps in a caller's workspace): read after a call of mla_decode_static on
// the same stream.  Copies 4 bytes to the host and synchronises the stream.
extern "C" mla_status mla_decode_static_status(int clear, mla_stream_t stream) {
  void* ws = nullptr;
  if (static_ws_address(&ws) != cudaSuccess) return MLA_ERR_CUDA;
  return mla_workspace_status(ws, clear, stream);
}
