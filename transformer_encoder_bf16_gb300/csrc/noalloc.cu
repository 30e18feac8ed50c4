// noalloc.cu -- laya_op_linear_noalloc: the tensor-core projection of
// laya_op_linear for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all, or cannot keep a workspace of
// their own: code that runs under a fixed device-memory budget owned by a host
// framework (whose allocator must not be bypassed), or a latency-critical loop
// where an allocation could synchronise the device or fail under a memory cap.
// The split-K plans of laya_op_linear need scratch memory for their partial
// tiles; this entry point takes it from a file-scope device array instead.
//
// The array is a fixed kNoallocScratchBytes (16 MiB) that every GPU loading
// this library holds until the process exits.  Host code cannot use the
// array's name as a device address, so the first call on each device looks
// the address up with cudaGetSymbolAddress (with that device current) and
// keeps it; make that first call before any stream capture.  Every call shares
// the array and leaves the last call's partial tiles in it: calls whose
// kernels overlap on the GPU (other streams, other host threads) race.
// Nothing in it has to start at zero: each call writes every partial it reads.
#include <mutex>

#include "../../include/laya_ops.h"
#include "internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = 16ull << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_split_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device); nullptr and the CUDA error on failure.
void* scratch_address(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_split_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

int laya_op_linear_noalloc(const void* x, int M, int K, const void* w, int N, int kind,
                           const void* residual, void* y, int splits, int tile_tokens,
                           void* stream) {
  if (!al16(x) || !al16(w) || !al16(y)) return LAYA_E_INVAL;
  if (kind == laya::kGemmResidual && !al16(residual)) return LAYA_E_INVAL;
  laya::GemmPlan p;
  if (!laya::plan_gemm(M, N, K, kind, laya::device_sm_count(), splits, tile_tokens, &p))
    return LAYA_E_INVAL;
  if (p.workspace_bytes > kNoallocScratchBytes) return LAYA_E_INVAL;  // beyond the fixed array
  laya::GemmOperands o;
  const uint64_t ldk = static_cast<uint64_t>(K) * 2;
  bool ok = laya::make_tmap_bf16_2d(&o.x, x, M, K, ldk, static_cast<uint32_t>(p.nt));
  if (kind == laya::kGemmGegluIl) {
    ok = ok && laya::make_tmap_geglu_il(&o.w, w, N, K);
    o.w2 = o.w;
  } else {
    ok = ok && laya::make_tmap_bf16_2d(&o.w, w, N, K, ldk, 128);
    if (kind == laya::kGemmGeglu) {
      const char* gate = static_cast<const char*>(w) + static_cast<size_t>(N) * K * 2;
      ok = ok && laya::make_tmap_bf16_2d(&o.w2, gate, N, K, ldk, 128);
    } else {
      o.w2 = o.w;
    }
  }
  if (!ok) return LAYA_E_INVAL;
  o.x_box_rows = p.x_box();
  o.y = static_cast<laya::bf16*>(y);
  o.residual = static_cast<const laya::bf16*>(residual);
  if (p.workspace_bytes > 0) {
    cudaError_t e = cudaSuccess;
    void* scratch = scratch_address(&e);
    if (scratch == nullptr) return LAYA_E_CUDA;
    o.partials = static_cast<float*>(scratch);
    o.partials_bytes = kNoallocScratchBytes;
  }
  laya::Launch l{static_cast<cudaStream_t>(stream), false};
  return laya::launch_gemm(p, o, l) == cudaSuccess ? LAYA_OK : LAYA_E_CUDA;
}

}  // extern "C"
