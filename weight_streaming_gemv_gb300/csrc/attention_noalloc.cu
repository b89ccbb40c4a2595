// Decode attention whose scratch is a fixed array inside this library, for
// callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a plugin running inside a host
// application that owns all device memory and hands it no allocator, a
// real-time loop in which an allocation's latency or an out-of-memory failure
// is not acceptable, or a process that reserved its device memory up front.
// qlin_attention_decode asks its caller for a workspace; this variant needs
// none.  Its chunk partials go to g_attn_scratch, a file-scope device array of
// QLIN_ATTENTION_NOALLOC_SCRATCH_BYTES (256 KiB), which every GPU that loads
// the library holds until the process exits.
#include <mutex>

#include "decode_ops.cuh"

namespace {

static __device__ __align__(256) float g_attn_scratch[QLIN_ATTENTION_NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
float *g_scratch_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device.  In host code the
// array's name only stands in for the symbol: a kernel given it would read the
// wrong memory or fault, so the address is looked up once per device, with
// that device current, and cached.
qlin_status scratch_of_current_device(float **out) {
    int dev = 0;
    QLIN_CUDA(cudaGetDevice(&dev));
    QLIN_REQUIRE(dev >= 0 && dev < kMaxDevices, QLIN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess || !p) {
            qlin::set_error("cudaGetSymbolAddress(g_attn_scratch) failed on device %d: %s", dev, cudaGetErrorString(e));
            return QLIN_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_addr[dev];
    return QLIN_OK;
}

}  // namespace

extern "C" qlin_status qlin_attention_decode_noalloc(const float *q, const float *k_cache, const float *v_cache,
                                                     int pos, int n_heads, int n_kv, int head_dim, float *out,
                                                     qlin_stream_t stream) {
    qlin::clear_error();
    QLIN_REQUIRE(q && k_cache && v_cache && out, QLIN_ERR_INVALID_ARG, "qlin_attention_decode_noalloc: null pointer");
    QLIN_REQUIRE(pos >= 0 && n_heads >= 1 && n_kv >= 1 && n_heads % n_kv == 0, QLIN_ERR_INVALID_ARG,
                 "qlin_attention_decode_noalloc: pos=%d n_heads=%d n_kv=%d", pos, n_heads, n_kv);
    QLIN_REQUIRE(head_dim >= 16 && head_dim <= 256 && (head_dim & (head_dim - 1)) == 0, QLIN_ERR_UNSUPPORTED,
                 "qlin_attention_decode_noalloc: head_dim %d", head_dim);
    QLIN_REQUIRE(pos < (1 << 20), QLIN_ERR_UNSUPPORTED, "qlin_attention_decode_noalloc: pos %d", pos);
    const size_t need = qlin_attention_workspace_size(pos + 1, n_heads, head_dim);
    QLIN_REQUIRE(need <= (size_t)QLIN_ATTENTION_NOALLOC_SCRATCH_BYTES, QLIN_ERR_UNSUPPORTED,
                 "qlin_attention_decode_noalloc: pos=%d, n_heads=%d, head_dim=%d need %zu bytes of scratch; the "
                 "library's fixed array holds %d (use qlin_attention_decode with a workspace instead)",
                 pos, n_heads, head_dim, need, QLIN_ATTENTION_NOALLOC_SCRATCH_BYTES);
    float *ws = nullptr;
    const qlin_status s = scratch_of_current_device(&ws);
    if (s) return s;
    return qlin::launch_attention(q, k_cache, v_cache, pos, n_heads, n_kv, head_dim, out, ws, (pos + 1 + 31) / 32,
                                  (cudaStream_t)stream);
}
