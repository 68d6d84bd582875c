// End-to-end box filter of host-resident sidecars (vbm_box_filter_batch_host,
// include/vbm.h): the grid owns two sets of device staging buffers and three
// streams (copies in, filter, copies out); each call copies its sidecars in,
// runs the batched box filter and copies the outputs back, with events
// ordering every reuse of a staging set, so that consecutive calls overlap.
// Host code only: the filter itself is the batched launcher of vbm_brick.cu
// (or the per-sidecar launchers of the other resolvers).
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "vbm_internal.h"
#include "vbm_launch.h"

namespace vbm {

struct HostIO {
    cudaStream_t s_in = nullptr, s_k = nullptr, s_out = nullptr;
    struct Set {
        char* dev = nullptr;  // sidecars, then outputs, each 256-byte aligned
        size_t bytes = 0;
        bool used = false;
        cudaEvent_t in_done = nullptr;   // the sidecars are on the device
        cudaEvent_t k_done = nullptr;    // the filter has read the sidecars and written the outputs
        cudaEvent_t out_done = nullptr;  // the outputs are back on the host
    } set[2];
    int next = 0;
};

void destroy_host_io(HostIO* h) {
    if (!h) return;
    for (cudaStream_t s : {h->s_in, h->s_k, h->s_out})
        if (s) cudaStreamSynchronize(s);
    for (HostIO::Set& S : h->set) {
        if (S.dev) cudaFree(S.dev);
        for (cudaEvent_t e : {S.in_done, S.k_done, S.out_done})
            if (e) cudaEventDestroy(e);
    }
    for (cudaStream_t s : {h->s_in, h->s_k, h->s_out})
        if (s) cudaStreamDestroy(s);
    delete h;
}

cudaError_t launch_box_batch(const DevGrid& g, int count, const float* const* sidecars, const int* C,
                             float* const* outs, int resolver, cudaStream_t stream) {
    cudaError_t e = cudaSuccess;
    if (g.n_blocks == 0) {
        for (int i = 0; i < count && e == cudaSuccess; ++i)
            e = cudaMemsetAsync(outs[i], 0, sizeof(float) * (size_t)C[i], stream);
    } else if (resolver == VBM_RESOLVE_BRICK) {
        e = launch_brick_box_batch(g, count, sidecars, C, outs, stream);
    } else {
        for (int i = 0; i < count && e == cudaSuccess; ++i)
            e = launch_box_filter(g, sidecars[i], C[i], outs[i], resolver, VBM_OUTPUT_STREAMED, stream);
    }
    return e;
}

namespace {

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

cudaError_t create_host_io(HostIO*& out) {
    HostIO* h = new HostIO;
    cudaError_t e = cudaSuccess;
    for (cudaStream_t* s : {&h->s_in, &h->s_k, &h->s_out})
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    for (HostIO::Set& S : h->set)
        for (cudaEvent_t* ev : {&S.in_done, &S.k_done, &S.out_done})
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        destroy_host_io(h);
        return e;
    }
    out = h;
    return cudaSuccess;
}

}  // namespace

int box_filter_batch_host(vbm_grid* g, int count, const float* const* host_sidecars, const int* C,
                          float* const* host_outs, int resolver, void* stream_v, std::string& err) {
    const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    std::lock_guard<std::mutex> lock(g->hostio_mu);
#define VBM_CK(call)                                                                                 \
    do {                                                                                             \
        const cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess) {                                                                     \
            cudaGetLastError();                                                                      \
            err = std::string("vbm_box_filter_batch_host: ") + #call + ": " + cudaGetErrorString(e_); \
            return VBM_ERR_CUDA;                                                                     \
        }                                                                                            \
    } while (0)
    if (!g->hostio) VBM_CK(create_host_io(g->hostio));
    HostIO& h = *g->hostio;
    size_t bytes[VBM_MAX_BATCH], off_in[VBM_MAX_BATCH], off_out[VBM_MAX_BATCH], total = 0;
    for (int i = 0; i < count; ++i) {
        bytes[i] = (size_t)(g->n + 1) * (size_t)C[i] * sizeof(float);
        off_in[i] = total;
        total += up256(bytes[i]);
    }
    for (int i = 0; i < count; ++i) {
        off_out[i] = total;
        total += up256(bytes[i]);
    }
    HostIO::Set& S = h.set[h.next];
    h.next ^= 1;
    if (S.bytes < total) {
        if (S.dev) {  // grow: wait for the set's last use, then replace it
            VBM_CK(cudaEventSynchronize(S.out_done));
            VBM_CK(cudaFree(S.dev));
            S.dev = nullptr;
            S.bytes = 0;
        }
        const cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&S.dev), total);
        if (e != cudaSuccess) {
            cudaGetLastError();
            S.dev = nullptr;
            err = "vbm_box_filter_batch_host: cudaMalloc of " + std::to_string(total) +
                  " bytes of staging failed: " + cudaGetErrorString(e);
            return VBM_ERR_NOMEM;
        }
        S.bytes = total;
        S.used = false;
    }
    const float* dev_in[VBM_MAX_BATCH];
    float* dev_out[VBM_MAX_BATCH];
    for (int i = 0; i < count; ++i) {
        dev_in[i] = reinterpret_cast<const float*>(S.dev + off_in[i]);
        dev_out[i] = reinterpret_cast<float*>(S.dev + off_out[i]);
    }
    // The sidecars in, once the set's previous filter has read its last ones.
    // Nothing orders this after the caller's stream: the host sidecars are
    // read as they are when the copies run (so that this call's copies overlap
    // the previous call's filter and copies back).
    if (S.used) VBM_CK(cudaStreamWaitEvent(h.s_in, S.k_done, 0));
    for (int i = 0; i < count; ++i)
        VBM_CK(cudaMemcpyAsync(S.dev + off_in[i], host_sidecars[i], bytes[i], cudaMemcpyHostToDevice, h.s_in));
    VBM_CK(cudaEventRecord(S.in_done, h.s_in));
    // The filter, once the sidecars are in and the set's previous outputs are out.
    VBM_CK(cudaStreamWaitEvent(h.s_k, S.in_done, 0));
    if (S.used) VBM_CK(cudaStreamWaitEvent(h.s_k, S.out_done, 0));
    VBM_CK(launch_box_batch(g->dev, count, dev_in, C, dev_out, resolver, h.s_k));
    VBM_CK(cudaEventRecord(S.k_done, h.s_k));
    // The outputs back; the caller's stream waits for them.
    VBM_CK(cudaStreamWaitEvent(h.s_out, S.k_done, 0));
    for (int i = 0; i < count; ++i)
        VBM_CK(cudaMemcpyAsync(host_outs[i], S.dev + off_out[i], bytes[i], cudaMemcpyDeviceToHost, h.s_out));
    VBM_CK(cudaEventRecord(S.out_done, h.s_out));
    VBM_CK(cudaStreamWaitEvent(stream, S.out_done, 0));
    S.used = true;
#undef VBM_CK
    return VBM_OK;
}

}  // namespace vbm
