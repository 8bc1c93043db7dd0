// Internal interface of the KV-cache decoder: the cache object and the persistent decode-step
// kernel (decode_mega.cu) that decode.cu launches when the shape and the device allow it.
#pragma once

#include "common.cuh"

struct gk_kv {
    gk_gpt_cfg cfg{};
    int B = 0, Tmax = 0;
    float* cache = nullptr;  // [L][2][B][H][Tmax][hs]
    int* state = nullptr;    // device: [0] cache length, [1] selections made
    int length = 0;          // host mirror of state[0]
    // activations (prefill uses B*Tmax rows, decode B rows)
    float *x = nullptr, *ln = nullptr, *qkv = nullptr, *y = nullptr, *pre = nullptr, *h = nullptr;
    float *mean = nullptr, *rstd = nullptr, *lse = nullptr, *last = nullptr;
    float* partial = nullptr;  // split-K partial sums
    size_t partial_floats = 0;
    float* attn_part = nullptr;  // decode attention partials [B*H][chunks][hs + 2]
    int* tickets = nullptr;      // last-block tickets: [0, 1024) GEMV column blocks, [1024, 2048) attention
    int32_t* ids = nullptr;      // gk_generate_uncached: the prefix [B, t] of each step, then next [B]
    // gk_decode_run: one captured decode step (instantiated graph) and what it was captured for
    cudaGraphExec_t graph = nullptr;
    int64_t graph_launches = 0;
    const void* graph_key[6] = {};
    gk_sample_cfg graph_s{};
    bool graph_has_s = false;
    // persistent decode step: grid barrier words (a 64-bit arrival count at [0], the abort word
    // at [32]) and whether this cache's shape runs it (decided at creation)
    unsigned* bar = nullptr;
    bool mega = false;
};

namespace gk {

// Set kv->mega if the persistent decode-step kernel takes this cache's shape on this device.
void mega_setup(gk_ctx* ctx, gk_kv* kv);
// Embedding, every layer (LayerNorm, QKV with the key/value append, attention, projection,
// MLP) and ln_f + the LM head of one decode step in one cooperative launch; logits [B, V].
gk_status mega_step(gk_ctx* ctx, gk_kv* kv, const float* params, const int32_t* tokens, float* logits);

}  // namespace gk
