// zero_host.cpp -- host-only entry points of libzero_gb300.so: the flat
// layout, the per-rank memory ledger, the communication count and status text.
//
// Sources: blog post "Data parallelism and ZeRO: how much each of the three
// stages saves", sections "16 bytes per parameter" and "three stages" (stage
// table); lecture deck "RC-T2", slide b1 and note N47; topic page "Putting the
// training ledger onto multiple devices", section "start from persistent
// state" (GB = 1e9 bytes, persistent state only).
#include <cstdint>

#include "zero_gb300.h"

namespace {

// Owners' slices have equal size only if the flat vector is padded to a
// multiple of N * ZERO_PAD_UNIT; the unit also keeps every slice a whole
// number of 16-byte vectors for BF16 and FP32 data.
int64_t round_up(int64_t x, int64_t unit) { return ((x + unit - 1) / unit) * unit; }

int64_t per_rank_share(int64_t psi, int32_t N) { return (psi + N - 1) / N; }

}  // namespace

extern "C" int zero_init_layout(const int64_t* tensor_numel, int64_t n_tensors, int32_t N,
                                zero_layout* out, int64_t* tensor_offsets) {
    if (out == nullptr || N < 1 || N > ZERO_MAX_RANKS || n_tensors < 0 ||
        (n_tensors > 0 && tensor_numel == nullptr))
        return ZERO_ERR_ARG;
    int64_t psi = 0;
    for (int64_t i = 0; i < n_tensors; ++i) {
        if (tensor_numel[i] < 0 || tensor_numel[i] > ZERO_MAX_ELEMS - psi) return ZERO_ERR_ARG;
        psi += tensor_numel[i];
    }
    if (psi > ZERO_MAX_ELEMS - static_cast<int64_t>(N) * ZERO_PAD_UNIT) return ZERO_ERR_ARG;
    // second pass writes the offsets only once every size is known to be valid
    if (tensor_offsets != nullptr) {
        int64_t at = 0;
        for (int64_t i = 0; i < n_tensors; ++i) {
            tensor_offsets[i] = at;
            at += tensor_numel[i];
        }
    }
    const int64_t unit = static_cast<int64_t>(N) * ZERO_PAD_UNIT;
    out->psi = psi;
    out->psi_pad = round_up(psi, unit);
    out->shard = out->psi_pad / N;
    out->n_tensors = n_tensors;
    out->N = N;
    out->pad_unit = ZERO_PAD_UNIT;
    return ZERO_OK;
}

extern "C" int zero_shard_range(const zero_layout* layout, int32_t r, int64_t* begin,
                                int64_t* end) {
    if (layout == nullptr || begin == nullptr || end == nullptr || r < 0 || r >= layout->N)
        return ZERO_ERR_ARG;
    *begin = static_cast<int64_t>(r) * layout->shard;
    *end = *begin + layout->shard;
    return ZERO_OK;
}

extern "C" int64_t zero_ledger(int64_t psi, int32_t N, int32_t stage, int32_t grad_bytes,
                               int32_t optim_bytes) {
    if (psi < 0 || psi > ZERO_MAX_ELEMS || N < 1 || grad_bytes < 0 || grad_bytes > 64 ||
        optim_bytes < 0 || optim_bytes > 64)
        return -1;
    const int64_t weight = 2;  // BF16 working weight
    const int64_t grad = grad_bytes;
    const int64_t optim = optim_bytes;
    const int64_t share = per_rank_share(psi, N);
    switch (stage) {
        case 0: return psi * (weight + grad + optim);                 // everything replicated
        case 1: return psi * (weight + grad) + share * optim;          // optimizer state sharded
        case 2: return psi * weight + share * (grad + optim);          // + gradients sharded
        case 3: return share * (weight + grad + optim);                // + working weights sharded
        default: return -1;
    }
}

extern "C" int64_t zero3_peak_bytes(const int64_t* layer_numel, int64_t n_layers, int32_t N,
                                   int32_t grad_bytes, int32_t optim_bytes) {
    if (n_layers < 0 || N < 1 || (n_layers > 0 && layer_numel == nullptr)) return -1;
    int64_t psi = 0;
    int64_t live = 0;  // the most elements alive in the two views at once
    for (int64_t i = 0; i < n_layers; ++i) {
        if (layer_numel[i] < 0 || layer_numel[i] > ZERO_MAX_ELEMS - psi) return -1;
        psi += layer_numel[i];
        const int64_t next = (i + 1 < n_layers) ? layer_numel[i + 1] : 0;
        if (layer_numel[i] + next > live) live = layer_numel[i] + next;
    }
    const int64_t persistent = zero_ledger(psi, N, 3, grad_bytes, optim_bytes);
    if (persistent < 0) return -1;
    return persistent + 2 * live;  // BF16 views
}

extern "C" int64_t zero_comm_volume(int64_t psi, int32_t N, int32_t stage) {
    if (psi < 0 || psi > ZERO_MAX_ELEMS || N < 1 || stage < 0 || stage > 3) return -1;
    // reduce-scatter + all-gather (= one all-reduce); ZeRO-3 gathers the
    // weights once more
    return (stage == 3 ? 3 : 2) * psi;
}

extern "C" const char* zero_status_str(int status) {
    switch (status) {
        case ZERO_OK: return "ok";
        case ZERO_STEP_SKIPPED: return "step skipped: non-finite gradient";
        case ZERO_ERR_ARG: return "invalid argument";
        case ZERO_ERR_ALIGN: return "buffer not 16-byte aligned";
        case ZERO_ERR_CUDA: return "CUDA error while enqueueing";
        case ZERO_ERR_TIMEOUT: return "bounded wait inside a kernel timed out";
        case ZERO_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case ZERO_ERR_OVERLAP: return "buffers that must be disjoint overlap";
        case ZERO_ERR_BOUNDS: return "index outside a buffer (debug build): access skipped";
        case ZERO_ERR_POLICY_WINDOW:
            return "device policy: the step's t fell outside its window of bias corrections";
        case ZERO_ERR_TOO_LARGE:
            return "step needs more scratch than the no-allocation entry point's fixed array";
        default: return "unknown status";
    }
}
