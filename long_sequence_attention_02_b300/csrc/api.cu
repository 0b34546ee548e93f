// C ABI of the library: argument checks, workspace sizing, RoPE tables, the
// device error word and launches. See include/wan_attn.h for the contract.
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.cuh"
#include "wan_attn.h"

namespace {

// A named NVTX range around a call's launches, so that profilers (nsys, or
// ncu --nvtx --nvtx-include "wan_attn_fwd/") can attribute and select them.
// With no tool attached, push and pop return at once.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

using wan::kHeadDim;

__device__ int g_wan_device_error;  // one per device that loads the library

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // 4 s per device-side wait

struct DeviceState {
  bool probed = false;
  bool supported = false;
  void* ctx = nullptr;  // the context the addresses below belong to
  int* err = nullptr;
  void* noalloc = nullptr;  // device address of the allocation-free scratch (looked up on first use)
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
int g_stall_launches = 0;
int g_check_launches = 0;     // wan_debug_inject_check
int g_last_check_line = 0;    // source line of the last debug check reported
uint64_t g_stall_timeout_ns = 0;
cudaEvent_t g_prof[wan::kNumPasses][2] = {};  // profiling hook, one-shot (guarded by g_mu)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int grid_tokens(wan_grid_t g, long long* L) {
  if (g.F <= 0 || g.Hp <= 0 || g.Wp <= 0) return WAN_ERR_INVALID;
  const long long l = (long long)g.F * g.Hp * g.Wp;
  if (l > INT_MAX) return WAN_ERR_INVALID;
  *L = l;
  return WAN_OK;
}

// Shape checks shared by the attention entry points (host only, no CUDA call).
int check_shapes(int B, long long L, int H, int head_dim) {
  if (B < 0 || H <= 0 || B > 65535 || H > 65535) return WAN_ERR_INVALID;
  if (head_dim != kHeadDim) return WAN_ERR_UNSUPPORTED;
  if ((unsigned long long)L * (unsigned long long)H >= (1ull << 31)) return WAN_ERR_INVALID;
  return WAN_OK;
}

// The current CUDA context (driver entry point fetched through the runtime,
// so the library needs no link-time dependency on libcuda). Device addresses
// of the library's __device__ symbols belong to a context: after a
// cudaDeviceReset (or any other re-creation of the primary context) the
// module is loaded again and they may move, so they are cached per context.
void* current_context() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  static GetCurrentFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCurrentFn>(p);
  }
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WAN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return WAN_ERR_UNSUPPORTED;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (st.probed && st.ctx != ctx) st = DeviceState();  // a new context: look the symbols up again
  if (!st.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return WAN_ERR_CUDA;
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_wan_device_error) != cudaSuccess) return WAN_ERR_CUDA;
      st.err = static_cast<int*>(p);
    }
    st.ctx = ctx;
    st.probed = true;
  }
  if (!st.supported) return WAN_ERR_UNSUPPORTED;
  *out = &st;
  return WAN_OK;
}

wan::LaunchCommon launch_common(const DeviceState& st) {
  wan::LaunchCommon lc;
  lc.err = st.err;
  lc.timeout_ns = kDefaultTimeoutNs;
  lc.stall = 0;
  lc.force_check = 0;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int p = 0; p < wan::kNumPasses; ++p)
    for (int i = 0; i < 2; ++i) {
      lc.ev[p][i] = g_prof[p][i];
      g_prof[p][i] = nullptr;
    }
  if (g_check_launches > 0) {
    --g_check_launches;
    lc.force_check = 1;
  }
  if (g_stall_launches > 0) {
    --g_stall_launches;
    lc.stall = 1;
    lc.timeout_ns = g_stall_timeout_ns;
  }
  return lc;
}

wan::RopeTables split_tables(const float* tables, wan_grid_t g) {
  wan::RopeTables t;
  const float2* base = reinterpret_cast<const float2*>(tables);
  t.t = base;
  t.h = base + (size_t)g.F * wan::kPairsT;
  t.w = t.h + (size_t)g.Hp * wan::kPairsH;
  return t;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Scratch of wan_attn_fwd_noalloc: the rotated keys of one call. Held on
// every device that loads the library; its device address is looked up once
// per device and context (noalloc_scratch below), since in host code the
// name is only a host-side stand-in.
static __device__ __align__(256) uint8_t g_wan_noalloc_scratch[WAN_NOALLOC_SCRATCH_BYTES];

// The scratch's device address for the current device and context (st from
// device_state, which resets it when the context changes).
int noalloc_scratch(DeviceState* st, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (st->noalloc == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wan_noalloc_scratch) != cudaSuccess || p == nullptr) return WAN_ERR_CUDA;
    st->noalloc = p;
  }
  *out = st->noalloc;
  return WAN_OK;
}

}  // namespace

extern "C" {

const char* wan_status_str(int status) {
  switch (status) {
    case WAN_OK: return "WAN_OK";
    case WAN_ERR_INVALID: return "WAN_ERR_INVALID: invalid argument";
    case WAN_ERR_UNSUPPORTED: return "WAN_ERR_UNSUPPORTED: head_dim or device not supported";
    case WAN_ERR_CUDA: return "WAN_ERR_CUDA: CUDA call or launch failed";
    case WAN_ERR_TIMEOUT: return "WAN_ERR_TIMEOUT: device-side wait expired";
    case WAN_ERR_DEVICE_CHECK: return "WAN_ERR_DEVICE_CHECK: a debug build's device-side check failed";
    default: return "unknown wan status";
  }
}

int wan_version(void) { return 100; }

size_t wan_rope3d_tables_size(wan_grid_t g, int head_dim) {
  long long L = 0;
  if (grid_tokens(g, &L) != WAN_OK || head_dim != kHeadDim) return 0;
  return ((size_t)g.F * wan::kPairsT + (size_t)g.Hp * wan::kPairsH + (size_t)g.Wp * wan::kPairsW) * 2 *
         sizeof(float);
}

int wan_rope3d_tables(wan_grid_t g, int head_dim, double theta, float* tables_dev, void* stream) {
  const NvtxRange nvtx_range("wan_rope3d_tables");
  long long L = 0;
  if (grid_tokens(g, &L) != WAN_OK) return WAN_ERR_INVALID;
  if (head_dim != kHeadDim) return WAN_ERR_UNSUPPORTED;
  if (tables_dev == nullptr || !(theta > 1.0) || !std::isfinite(theta)) return WAN_ERR_INVALID;
  // Bands t, h, w of widths 44, 42, 42: pair j of a band of width w turns by
  // pos * theta^(-2j / w), evaluated in double precision.
  const int widths[3] = {2 * wan::kPairsT, 2 * wan::kPairsH, 2 * wan::kPairsW};
  const int npos[3] = {g.F, g.Hp, g.Wp};
  std::vector<float> host;
  host.reserve(wan_rope3d_tables_size(g, head_dim) / sizeof(float));
  for (int ax = 0; ax < 3; ++ax) {
    const int pairs = widths[ax] / 2;
    for (int pos = 0; pos < npos[ax]; ++pos)
      for (int j = 0; j < pairs; ++j) {
        const double omega = std::pow(theta, -2.0 * j / widths[ax]);
        const double ang = (double)pos * omega;
        host.push_back((float)std::cos(ang));
        host.push_back((float)std::sin(ang));
      }
  }
  cudaError_t e = cudaMemcpyAsync(tables_dev, host.data(), host.size() * sizeof(float), cudaMemcpyHostToDevice,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

size_t wan_attn_workspace_size(int op, int B, wan_grid_t g, int H, int head_dim) {
  long long L = 0;
  if (grid_tokens(g, &L) != WAN_OK || check_shapes(B, L, H, head_dim) != WAN_OK) return 0;
  if (op == WAN_OP_FWD) return round_up((size_t)B * L * H * kHeadDim * 2, 256);
  if (op == WAN_OP_BWD) return wan::attn_bwd_workspace_bytes(B, (int)L, H);
  if (op == WAN_OP_FWD_FP8) return wan::attn_fwd_fp8_workspace_bytes(B, (int)L, H);
  return 0;
}

int wan_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g, int H,
                 int head_dim, const float* tables, float scale, void* workspace, size_t ws_bytes,
                 void* stream) {
  const NvtxRange nvtx_range("wan_attn_fwd");
  long long L = 0;
  int rc = grid_tokens(g, &L);
  if (rc == WAN_OK) rc = check_shapes(B, L, H, head_dim);
  if (rc != WAN_OK) return rc;
  if (!q || !k || !v || !o || !tables || !workspace) return B == 0 ? WAN_OK : WAN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(tables) & 7u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return WAN_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return WAN_ERR_INVALID;
  if (ws_bytes < wan_attn_workspace_size(WAN_OP_FWD, B, g, H, head_dim)) return WAN_ERR_INVALID;
  if (B == 0) return WAN_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != WAN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const wan::RopeTables tab = split_tables(tables, g);
  const wan::LaunchCommon lc = launch_common(*st);
  {
    const NvtxRange pass("k_rotate");
    wan::record_pass(lc, wan::kPassRope, 0, s);
    if (wan::launch_rope_rotate_bf16(k, workspace, B, g, H, tab, false, s) != cudaSuccess) return WAN_ERR_CUDA;
    wan::record_pass(lc, wan::kPassRope, 1, s);
  }
  const NvtxRange pass("attention");
  return wan::launch_attn_fwd(q, workspace, v, o, lse, B, (int)L, (int)L, H, g, tab, true, nullptr, scale, lc, s);
}

int wan_xattn_fwd(const void* q, const void* k, const void* v, const int32_t* kv_lens, int Lk, void* o,
                  float* lse, int B, wan_grid_t g, int H, int head_dim, float scale, void* stream) {
  const NvtxRange nvtx_range("wan_xattn_fwd");
  long long L = 0;
  int rc = grid_tokens(g, &L);
  if (rc == WAN_OK) rc = check_shapes(B, L, H, head_dim);
  if (rc != WAN_OK) return rc;
  if (Lk < 1 || Lk > 512) return WAN_ERR_INVALID;
  if (!q || !k || !v || !o) return B == 0 ? WAN_OK : WAN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(kv_lens) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return WAN_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return WAN_ERR_INVALID;
  if (B == 0) return WAN_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != WAN_OK) return rc;
  return wan::launch_attn_fwd(q, k, v, o, lse, B, (int)L, Lk, H, g, wan::RopeTables{}, false, kv_lens, scale,
                              launch_common(*st), static_cast<cudaStream_t>(stream));
}

int wan_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, wan_grid_t g, int H, int head_dim, const float* tables,
                 float scale, void* workspace, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx_range("wan_attn_bwd");
  long long L = 0;
  int rc = grid_tokens(g, &L);
  if (rc == WAN_OK) rc = check_shapes(B, L, H, head_dim);
  if (rc != WAN_OK) return rc;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !tables || !workspace)
    return B == 0 ? WAN_OK : WAN_ERR_INVALID;
  const void* ptrs[10] = {q, k, v, o, dout, dq, dk, dv, workspace, lse};
  for (const void* p : ptrs)
    if (!aligned16(p)) return WAN_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(tables) & 7u) return WAN_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return WAN_ERR_INVALID;
  if (ws_bytes < wan_attn_workspace_size(WAN_OP_BWD, B, g, H, head_dim)) return WAN_ERR_INVALID;
  if (B == 0) return WAN_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != WAN_OK) return rc;
  return wan::launch_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, g, H, split_tables(tables, g), scale,
                              workspace, launch_common(*st), static_cast<cudaStream_t>(stream));
}

int wan_attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g, int H,
                     int head_dim, const float* tables, float scale, void* workspace, size_t ws_bytes,
                     void* stream) {
  const NvtxRange nvtx_range("wan_attn_fwd_fp8");
  long long L = 0;
  int rc = grid_tokens(g, &L);
  if (rc == WAN_OK) rc = check_shapes(B, L, H, head_dim);
  if (rc != WAN_OK) return rc;
  if (!q || !k || !v || !o || !tables || !workspace) return B == 0 ? WAN_OK : WAN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(tables) & 7u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return WAN_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return WAN_ERR_INVALID;
  if (ws_bytes < wan_attn_workspace_size(WAN_OP_FWD_FP8, B, g, H, head_dim)) return WAN_ERR_INVALID;
  if (B == 0) return WAN_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != WAN_OK) return rc;
  return wan::launch_attn_fwd_fp8(q, k, v, o, lse, B, g, H, split_tables(tables, g), scale, workspace,
                                  launch_common(*st), static_cast<cudaStream_t>(stream));
}

int wan_attn_fwd_ring_step(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g,
                           int H, int head_dim, const float* tables, float scale, int q_start, int q_len,
                           int kv_start, int kv_len, int accumulate, void* workspace, size_t ws_bytes,
                           void* stream) {
  const NvtxRange nvtx_range("wan_attn_fwd_ring_step");
  long long L = 0;
  int rc = grid_tokens(g, &L);
  if (rc == WAN_OK) rc = check_shapes(B, L, H, head_dim);
  if (rc != WAN_OK) return rc;
  if (q_start < 0 || q_len < 1 || (long long)q_start + q_len > L || kv_start < 0 || kv_len < 1 ||
      (long long)kv_start + kv_len > L || (accumulate != 0 && accumulate != 1))
    return WAN_ERR_INVALID;
  if (!q || !k || !v || !o || !lse || !tables || !workspace) return B == 0 ? WAN_OK : WAN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(tables) & 7u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return WAN_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return WAN_ERR_INVALID;
  if (ws_bytes < round_up((size_t)B * kv_len * H * kHeadDim * 2, 256)) return WAN_ERR_INVALID;
  if (B == 0) return WAN_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != WAN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const wan::RopeTables tab = split_tables(tables, g);
  const wan::LaunchCommon lc = launch_common(*st);
  {
    const NvtxRange pass("k_rotate");
    wan::record_pass(lc, wan::kPassRope, 0, s);
    if (wan::launch_rope_rotate_bf16_rows(k, workspace, B, kv_len, kv_start, g, H, tab, false, s) != cudaSuccess)
      return WAN_ERR_CUDA;
    wan::record_pass(lc, wan::kPassRope, 1, s);
  }
  const NvtxRange pass("attention");
  return wan::launch_attn_fwd(q, workspace, v, o, lse, B, q_len, kv_len, H, g, tab, true, nullptr, scale, lc, s,
                              q_start, accumulate ? wan::kMergeLse : wan::kMergeNone);
}

int wan_xattn_fwd_dual(const void* q, const void* k_txt, const void* v_txt, const int32_t* lens_txt, int Lk_txt,
                       const void* k_img, const void* v_img, const int32_t* lens_img, int Lk_img, void* o,
                       float* lse, int B, wan_grid_t g, int H, int head_dim, float scale, void* stream) {
  const NvtxRange nvtx_range("wan_xattn_fwd_dual");
  long long L = 0;
  int rc = grid_tokens(g, &L);
  if (rc == WAN_OK) rc = check_shapes(B, L, H, head_dim);
  if (rc != WAN_OK) return rc;
  if (Lk_txt < 1 || Lk_txt > 512 || Lk_img < 1 || Lk_img > 512) return WAN_ERR_INVALID;
  if (!q || !k_txt || !v_txt || !k_img || !v_img || !o) return B == 0 ? WAN_OK : WAN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_txt) || !aligned16(v_txt) || !aligned16(k_img) || !aligned16(v_img) ||
      !aligned16(o) || (reinterpret_cast<uintptr_t>(lens_txt) & 3u) || (reinterpret_cast<uintptr_t>(lens_img) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return WAN_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return WAN_ERR_INVALID;
  if (B == 0) return WAN_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != WAN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = wan::launch_attn_fwd(q, k_txt, v_txt, o, lse, B, (int)L, Lk_txt, H, g, wan::RopeTables{}, false, lens_txt,
                            scale, launch_common(*st), s);
  if (rc != WAN_OK) return rc;
  return wan::launch_attn_fwd(q, k_img, v_img, o, nullptr, B, (int)L, Lk_img, H, g, wan::RopeTables{}, false,
                              lens_img, scale, launch_common(*st), s, 0, wan::kMergeAdd);
}

int wan_get_device_status(void* stream) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != WAN_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return WAN_ERR_CUDA;
  int v = 0;
  const int zero = 0;
  if (cudaMemcpy(&v, st->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return WAN_ERR_CUDA;
  if (v != 0 && cudaMemcpy(st->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return WAN_ERR_CUDA;
  if ((v & 0xFF) == wan::kDevCheck) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_last_check_line = v >> 8;
    return WAN_ERR_DEVICE_CHECK;
  }
  return v == 0 ? WAN_OK : v;
}

int wan_profile_set_pass_events(int pass, void* start, void* stop) {
  if (pass < 0 || pass >= wan::kNumPasses || (start == nullptr) != (stop == nullptr)) return WAN_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  g_prof[pass][0] = static_cast<cudaEvent_t>(start);
  g_prof[pass][1] = static_cast<cudaEvent_t>(stop);
  return WAN_OK;
}

int wan_profile_set_events(void* start, void* stop) { return wan_profile_set_pass_events(WAN_PASS_MAIN, start, stop); }

int wan_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g,
                         int H, int head_dim, const float* tables, float scale, void* stream) {
  const NvtxRange nvtx_range("wan_attn_fwd_noalloc");
  long long L = 0;
  int rc = grid_tokens(g, &L);
  if (rc == WAN_OK) rc = check_shapes(B, L, H, head_dim);
  if (rc != WAN_OK) return rc;
  // The rotated keys (B * L * H rows of 256 bytes) must fit the fixed scratch.
  if ((unsigned long long)B * (unsigned long long)L * (unsigned long long)H > WAN_NOALLOC_MAX_ROW_HEADS)
    return WAN_ERR_INVALID;
  if (B == 0) return WAN_OK;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != WAN_OK) return rc;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(st, &scratch)) != WAN_OK) return rc;
  return wan_attn_fwd(q, k, v, o, lse, B, g, H, head_dim, tables, scale, scratch, WAN_NOALLOC_SCRATCH_BYTES,
                      stream);
}

int wan_vae_causal_conv3d(const void* x, const void* cache, const void* weight, const float* bias, void* y,
                          void* cache_out, int B, int T, int H, int W, int c_in, int c_out, void* stream) {
  const NvtxRange nvtx_range("wan_vae_causal_conv3d");
  if (B < 0 || T <= 0 || H <= 0 || W <= 0 || c_in <= 0 || c_out <= 0 || B > 65535 || T > 65535 || H > 65535 ||
      W > 65535)
    return WAN_ERR_INVALID;
  if (c_in % 32 != 0 || c_in > 8192 || c_out > 8192 || wan::conv3d_n_tile(c_out) == 0) return WAN_ERR_UNSUPPORTED;
  if (B == 0) return WAN_OK;
  if (!x || !weight || !y) return WAN_ERR_INVALID;
  if (!aligned16(x) || !aligned16(weight) || !aligned16(y) || (cache && !aligned16(cache)) ||
      (cache_out && !aligned16(cache_out)) || (reinterpret_cast<uintptr_t>(bias) & 3u))
    return WAN_ERR_INVALID;
  const size_t frame = (size_t)H * W * c_in * 2;  // bytes of one input frame
  const size_t x_bytes = (size_t)B * T * frame, c_bytes = (size_t)B * 2 * frame;
  const size_t y_bytes = (size_t)B * T * H * W * c_out * 2, w_bytes = (size_t)c_out * 27 * c_in * 2;
  auto overlap = [](const void* p, size_t n, const void* q, size_t m) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return p && q && a < b + m && b < a + n;
  };
  if (overlap(y, y_bytes, x, x_bytes) || overlap(y, y_bytes, weight, w_bytes) || overlap(y, y_bytes, cache, c_bytes) ||
      overlap(cache_out, c_bytes, x, x_bytes) || overlap(cache_out, c_bytes, y, y_bytes) ||
      (cache_out != cache && overlap(cache_out, c_bytes, cache, c_bytes)))
    return WAN_ERR_INVALID;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != WAN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = wan::launch_causal_conv3d(x, cache, weight, bias, y, B, T, H, W, c_in, c_out, launch_common(*st), s);
  if (rc != WAN_OK || cache_out == nullptr) return rc;
  // Next chunk's cache: the last two frames of (cache or zeros) ++ x. Issued
  // after the convolution, so cache_out may be the cache it has just read.
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  const uint8_t* cb = static_cast<const uint8_t*>(cache);
  uint8_t* ob = static_cast<uint8_t*>(cache_out);
  for (int b = 0; b < B; ++b) {
    uint8_t* dst = ob + (size_t)b * 2 * frame;
    const uint8_t* xs = xb + (size_t)b * T * frame;
    cudaError_t e;
    if (T >= 2) {
      e = cudaMemcpyAsync(dst, xs + (size_t)(T - 2) * frame, 2 * frame, cudaMemcpyDeviceToDevice, s);
    } else {
      e = cb ? cudaMemcpyAsync(dst, cb + ((size_t)b * 2 + 1) * frame, frame, cudaMemcpyDeviceToDevice, s)
             : cudaMemsetAsync(dst, 0, frame, s);
      if (e == cudaSuccess) e = cudaMemcpyAsync(dst + frame, xs, frame, cudaMemcpyDeviceToDevice, s);
    }
    if (e != cudaSuccess) return WAN_ERR_CUDA;
  }
  return WAN_OK;
}

int wan_vae_time_downsample(const void* x, const void* cache, const void* weight, const float* bias, void* y,
                            void* cache_out, int B, int T, int H, int W, int c_in, int c_out, void* stream) {
  const NvtxRange nvtx_range("wan_vae_time_downsample");
  if (B < 0 || T <= 0 || H <= 0 || W <= 0 || c_in <= 0 || c_out <= 0 || B > 65535 || T > 65535 || H > 65535 ||
      W > 65535)
    return WAN_ERR_INVALID;
  // A first chunk is one frame and passes through; later chunks are even.
  if (cache ? T % 2 != 0 : (T != 1 || c_out != c_in)) return WAN_ERR_INVALID;
  if (c_in % 32 != 0 || c_in > 8192 || c_out > 8192 || wan::conv3d_n_tile(c_out) == 0) return WAN_ERR_UNSUPPORTED;
  if (B == 0) return WAN_OK;
  if (!x || !y || (cache && !weight)) return WAN_ERR_INVALID;
  if (!aligned16(x) || !aligned16(y) || (weight && !aligned16(weight)) || (cache && !aligned16(cache)) ||
      (cache_out && !aligned16(cache_out)) || (reinterpret_cast<uintptr_t>(bias) & 3u))
    return WAN_ERR_INVALID;
  const size_t frame = (size_t)H * W * c_in * 2;  // bytes of one input frame
  const int t_out = cache ? T / 2 : 1;
  const size_t x_bytes = (size_t)B * T * frame, c_bytes = (size_t)B * frame;
  const size_t y_bytes = (size_t)B * t_out * H * W * c_out * 2, w_bytes = (size_t)c_out * 3 * c_in * 2;
  auto overlap = [](const void* p, size_t n, const void* q, size_t m) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return p && q && a < b + m && b < a + n;
  };
  if (overlap(y, y_bytes, x, x_bytes) || (cache && overlap(y, y_bytes, weight, w_bytes)) ||
      overlap(y, y_bytes, cache, c_bytes) || overlap(cache_out, c_bytes, x, x_bytes) ||
      overlap(cache_out, c_bytes, y, y_bytes) || (cache_out != cache && overlap(cache_out, c_bytes, cache, c_bytes)))
    return WAN_ERR_INVALID;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc != WAN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cache) {
    rc = wan::launch_causal_conv3d(x, cache, weight, bias, y, B, T, H, W, c_in, c_out, launch_common(*st), s,
                                   /*time_down=*/true);
    if (rc != WAN_OK) return rc;
  } else if (cudaMemcpyAsync(y, x, x_bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess) {
    return WAN_ERR_CUDA;
  }
  if (cache_out == nullptr) return WAN_OK;
  // Next chunk's cache: the chunk's last input frame, written after the
  // convolution has read cache (cache_out may be that buffer).
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  uint8_t* ob = static_cast<uint8_t*>(cache_out);
  if (T == 1)
    return cudaMemcpyAsync(ob, xb, x_bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
  for (int b = 0; b < B; ++b)
    if (cudaMemcpyAsync(ob + (size_t)b * frame, xb + ((size_t)b * T + T - 1) * frame, frame,
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return WAN_ERR_CUDA;
  return WAN_OK;
}

int wan_debug_build(void) {
#ifdef WAN_DEBUG
  return 1;
#else
  return 0;
#endif
}

int wan_debug_inject_check(int count) {
  if (count < 0) return WAN_ERR_INVALID;
  if (!wan_debug_build()) return WAN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  g_check_launches = count;
  return WAN_OK;
}

int wan_debug_check_line(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_last_check_line;
}

int wan_debug_inject_stall(int count, int timeout_ms) {
  if (count < 0 || timeout_ms < 1 || timeout_ms > 10000) return WAN_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  g_stall_launches = count;
  g_stall_timeout_ns = (uint64_t)timeout_ms * 1000000ull;
  return WAN_OK;
}

}  // extern "C"
