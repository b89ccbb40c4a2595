// Host side of the qlin C ABI: status strings, thread-local error text,
// device attributes and the T158 packing of "Gemma 3 1B at 114 tokens per
// second on a laptop CPU", "Step 1: a kernel for 1.6-bit weights".
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <vector>

#include "common.cuh"

namespace qlin {

static thread_local std::string g_err;

void set_error(const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
}

void clear_error() { g_err.clear(); }

namespace {
struct DevAttr {
    int sms = 0, smem_optin = 0;
};
std::mutex g_attr_mu;
std::vector<DevAttr> g_attr;

DevAttr attr_of_current() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DevAttr{};
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if ((int)g_attr.size() <= dev) g_attr.resize(dev + 1);
    DevAttr &a = g_attr[dev];
    if (a.sms == 0) {
        cudaDeviceGetAttribute(&a.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&a.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    }
    return a;
}
}  // namespace

int sm_count() {
    int s = attr_of_current().sms;
    return s > 0 ? s : 1;
}

int max_smem_optin() { return attr_of_current().smem_optin; }

namespace {
std::mutex g_occ_mu;
std::map<std::tuple<const void *, int, size_t>, int> g_occ;
std::set<std::pair<const void *, int>> g_attr_set;
}  // namespace

int blocks_per_sm(const void *kern, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    auto key = std::make_tuple(kern, dev, smem);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
    if (!g_attr_set.count({kern, dev})) {
        // dynamic + static shared memory may not exceed the opt-in limit
        cudaFuncAttributes fa{};
        const int optin = attr_of_current().smem_optin;
        if (cudaFuncGetAttributes(&fa, kern) == cudaSuccess && optin > 48 * 1024)
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
        g_attr_set.insert({kern, dev});
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 256, smem) != cudaSuccess || n < 1) n = 1;
    g_occ[key] = n;
    return n;
}

}  // namespace qlin

extern "C" {

const char *qlin_status_str(int s) {
    switch (s) {
        case QLIN_OK: return "QLIN_OK";
        case QLIN_ERR_INVALID_ARG: return "QLIN_ERR_INVALID_ARG";
        case QLIN_ERR_UNSUPPORTED: return "QLIN_ERR_UNSUPPORTED";
        case QLIN_ERR_BAD_PACKED: return "QLIN_ERR_BAD_PACKED";
        case QLIN_ERR_CUDA: return "QLIN_ERR_CUDA";
        case QLIN_ERR_TIMEOUT: return "QLIN_ERR_TIMEOUT";
        default: return "QLIN_ERR_UNKNOWN";
    }
}

const char *qlin_last_error(void) { return qlin::g_err.c_str(); }

int qlin_version(void) { return 100; }

int64_t t158_pitch(int64_t K) {
    if (K < 1) return 0;
    const int64_t bytes = (K + 4) / 5;
    return (bytes + 15) / 16 * 16;
}

qlin_status t158_pack(const int8_t *trits, int64_t N, int64_t K, uint8_t *packed, int64_t pitch) {
    qlin::clear_error();
    QLIN_REQUIRE(trits && packed, QLIN_ERR_INVALID_ARG, "t158_pack: null pointer");
    QLIN_REQUIRE(N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "t158_pack: N=%lld K=%lld", (long long)N, (long long)K);
    QLIN_REQUIRE(pitch >= (K + 4) / 5, QLIN_ERR_INVALID_ARG, "t158_pack: pitch %lld < ceil(K/5)", (long long)pitch);
    for (int64_t i = 0; i < N * K; i++)
        QLIN_REQUIRE(trits[i] >= -1 && trits[i] <= 1, QLIN_ERR_INVALID_ARG, "t158_pack: trit %d at %lld",
                     (int)trits[i], (long long)i);
    const int64_t full = K / 5;  // bytes whose five trits are all < K
    for (int64_t n = 0; n < N; n++) {
        const int8_t *t = trits + n * K;
        uint8_t *row = packed + n * pitch;
        for (int64_t j = 0; j < full; j++) {
            const int8_t *g = t + 5 * j;
            row[j] = (uint8_t)((g[0] + 1) + 3 * (g[1] + 1) + 9 * (g[2] + 1) + 27 * (g[3] + 1) + 81 * (g[4] + 1));
        }
        for (int64_t j = full; j < pitch; j++) {
            int v = 0, p3 = 1;
            for (int i = 0; i < 5; i++, p3 *= 3) {
                const int64_t k = 5 * j + i;
                v += p3 * (k < K ? t[k] + 1 : 1);
            }
            row[j] = (uint8_t)v;
        }
    }
    return QLIN_OK;
}

int64_t t158_group_pitch(int64_t N) { return N < 1 ? 0 : (N + 15) / 16 * 16; }

qlin_status t158_pack_groups(const int8_t *trits, int64_t N, int64_t K, uint8_t *packed_g, int64_t gpitch) {
    qlin::clear_error();
    QLIN_REQUIRE(trits && packed_g, QLIN_ERR_INVALID_ARG, "t158_pack_groups: null pointer");
    QLIN_REQUIRE(N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "t158_pack_groups: N=%lld K=%lld", (long long)N,
                 (long long)K);
    QLIN_REQUIRE(gpitch >= N, QLIN_ERR_INVALID_ARG, "t158_pack_groups: gpitch %lld < N", (long long)gpitch);
    for (int64_t i = 0; i < N * K; i++)
        QLIN_REQUIRE(trits[i] >= -1 && trits[i] <= 1, QLIN_ERR_INVALID_ARG, "t158_pack_groups: trit %d at %lld",
                     (int)trits[i], (long long)i);
    const int64_t G = (K + 3) / 4;
    for (int64_t g = 0; g < G; g++) {
        uint8_t *dst = packed_g + g * gpitch;
        for (int64_t n = 0; n < N; n++) {
            const int8_t *t = trits + n * K + 4 * g;
            int v = 0, p3 = 1;
            for (int i = 0; i < 4; i++, p3 *= 3) v += p3 * (4 * g + i < K ? t[i] + 1 : 1);
            dst[n] = (uint8_t)v;
        }
        for (int64_t n = N; n < gpitch; n++) dst[n] = 40;  // four zero trits
    }
    return QLIN_OK;
}

qlin_status t158_unpack(const uint8_t *packed, int64_t N, int64_t K, int64_t pitch, int8_t *trits) {
    qlin::clear_error();
    QLIN_REQUIRE(trits && packed, QLIN_ERR_INVALID_ARG, "t158_unpack: null pointer");
    QLIN_REQUIRE(N >= 1 && K >= 1, QLIN_ERR_INVALID_ARG, "t158_unpack: N=%lld K=%lld", (long long)N, (long long)K);
    QLIN_REQUIRE(pitch >= (K + 4) / 5, QLIN_ERR_INVALID_ARG, "t158_unpack: pitch %lld < ceil(K/5)", (long long)pitch);
    for (int64_t i = 0; i < N * pitch; i++)
        QLIN_REQUIRE(packed[i] <= 242, QLIN_ERR_BAD_PACKED, "t158_unpack: byte %d at offset %lld", (int)packed[i],
                     (long long)i);
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) {
            int v = packed[n * pitch + k / 5];
            for (int64_t i = 0; i < k % 5; i++) v /= 3;
            trits[n * K + k] = (int8_t)(v % 3 - 1);
        }
    return QLIN_OK;
}

}  // extern "C"
