/*
 * example.c -- one MoE layer call through the C ABI of moe.h.
 *
 * The weights are device buffers laid out as moe.h describes; the caller owns
 * them and the workspace. Build:
 *   gcc -std=c11 -I include -I $CUDA_HOME/include example.c \
 *       -L token_dispatch_grouped_moe_gb300 -lmoe_gb300 -L $CUDA_HOME/lib64 -lcudart
 */
#include <cuda_runtime.h>

#include "moe.h"

/* One Mixtral-shaped layer call on `stream`; x, Wg, W1, W3, W2 and out are
 * device pointers. Returns a moe_status. */
int moe_forward(const moe_bf16* x, const moe_bf16* Wg, const moe_bf16* W1, const moe_bf16* W3,
                const moe_bf16* W2, moe_bf16* out, int64_t T, cudaStream_t stream)
{
    moe_dims d = {T, 4096, 14336, 8, 2, 0}; /* T tokens, H, F, E, top-k, no shared expert */
    size_t ws_bytes = moe_workspace_size(&d);
    void* ws = NULL;
    if (cudaMalloc(&ws, ws_bytes) != cudaSuccess) return MOE_ERR_CUDA;
    moe_status st = moe_layer_forward(&d, x, Wg, NULL, W1, W3, W2, NULL, NULL, NULL, out, NULL, ws,
                                      ws_bytes, NULL, (moe_stream_t)stream);
    if (st == MOE_OK) st = moe_check(ws, (moe_stream_t)stream); /* synchronises */
    cudaFree(ws);
    return st;
}

#ifdef MOE_EXAMPLE_MAIN
int main(void) { return 0; }
#endif
