// Decode attention that allocates nothing: the split-K flash-decode kernels
// of k_attn.cu, launched with their partial results in a file-scope device
// array instead of memory the engine obtained from cudaMalloc.
//
// Who needs this: code that may not allocate device memory on its own — a
// plug-in running under a host framework that owns every allocation, or a
// real-time audio thread that must not block in the allocator. Such callers
// bring their own inputs and outputs and get the scratch from this fixed
// array.
#include <mutex>

#include "common.cuh"
#include "../../include/tts_bb.h"

namespace {

using namespace ttsbb;

constexpr int STATIC_MAX_B = TTS_BB_STATIC_ATTN_MAX_B;
constexpr int STATIC_MAX_SPLITS = TTS_BB_STATIC_ATTN_MAX_SPLITS;
constexpr int MAX_DEVICES = 64;

// Split partials: [B][16 heads][splits][128 outputs + running max + running sum].
// Every GPU that loads the library holds this array (4.26 MB) until exit.
static __device__ __align__(256) float g_attn_scratch[(size_t)STATIC_MAX_B * NQ * STATIC_MAX_SPLITS * (HD + 2)];
// Page-table row of sequence b is row b: the identity map 0..STATIC_MAX_B-1.
static __device__ __align__(256) int32_t g_seq_rows[STATIC_MAX_B] = {
    0,  1,  2,  3,  4,  5,  6,  7,  8,  9,  10, 11, 12, 13, 14, 15, 16, 17, 18, 19, 20, 21,
    22, 23, 24, 25, 26, 27, 28, 29, 30, 31, 32, 33, 34, 35, 36, 37, 38, 39, 40, 41, 42, 43,
    44, 45, 46, 47, 48, 49, 50, 51, 52, 53, 54, 55, 56, 57, 58, 59, 60, 61, 62, 63};
static_assert(STATIC_MAX_B == 64, "g_seq_rows lists 64 rows");
// Query positions clamped into 0..max_position, so that no sequence reads a
// page-table entry past its row or a block the caller did not map.
static __device__ __align__(256) int32_t g_pos[STATIC_MAX_B];

__global__ void k_clamp_positions(const int32_t* __restrict__ positions, int B, int max_position) {
    const int b = threadIdx.x;
    if (b < B) g_pos[b] = min(max(positions[b], 0), max_position);
}

struct DeviceAddrs {
    float* scratch = nullptr;
    int32_t* rows = nullptr;
    int32_t* pos = nullptr;
    bool ready = false;
};
DeviceAddrs g_addrs[MAX_DEVICES];
std::mutex g_mu;

// Device addresses of the three arrays for the current device. In host code the
// array names are host-side stand-ins, not device addresses, so they are
// looked up once per device with that device current.
tts_bb_status device_addrs(DeviceAddrs** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return TTS_BB_E_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceAddrs& a = g_addrs[dev];
    if (!a.ready) {
        void* s = nullptr;
        void* r = nullptr;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&s, g_attn_scratch) != cudaSuccess) return TTS_BB_E_CUDA;
        if (cudaGetSymbolAddress(&r, g_seq_rows) != cudaSuccess) return TTS_BB_E_CUDA;
        if (cudaGetSymbolAddress(&p, g_pos) != cudaSuccess) return TTS_BB_E_CUDA;
        a.scratch = static_cast<float*>(s);
        a.rows = static_cast<int32_t*>(r);
        a.pos = static_cast<int32_t*>(p);
        a.ready = true;
    }
    *out = &a;
    return TTS_BB_OK;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) tts_bb_status tts_bb_gqa_decode_attention_static(
    const void* q, const void* kv_pool, const int32_t* page_table, int blocks_per_seq, const int32_t* positions,
    int B, int max_position, void* out, void* stream) {
    if (!q || !kv_pool || !page_table || !positions || !out) return TTS_BB_E_INVALID;
    if (B < 1 || B > STATIC_MAX_B) return TTS_BB_E_INVALID;  // beyond the fixed scratch
    // 64-bit, so that a max_position near INT_MAX cannot wrap past the check
    if (blocks_per_seq < 1 || max_position < 0 || (long long)max_position + 1 > (long long)blocks_per_seq * KVB)
        return TTS_BB_E_INVALID;
    DeviceAddrs* a = nullptr;
    const tts_bb_status s = device_addrs(&a);
    if (s != TTS_BB_OK) return s;
    // an error left pending by earlier work would otherwise be reported as this call's
    if (cudaPeekAtLastError() != cudaSuccess) return TTS_BB_E_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    k_clamp_positions<<<1, STATIC_MAX_B, 0, st>>>(positions, B, max_position);
    if (cudaPeekAtLastError() != cudaSuccess) return TTS_BB_E_CUDA;
    KVView kv{const_cast<bf16*>(static_cast<const bf16*>(kv_pool)), page_table, a->rows, blocks_per_seq};
    launch_attn_decode(static_cast<const bf16*>(q), kv, a->pos, B, max_position + 1, a->scratch,
                       static_cast<bf16*>(out), STATIC_MAX_SPLITS, st);
    return cudaPeekAtLastError() == cudaSuccess ? TTS_BB_OK : TTS_BB_E_CUDA;
}
