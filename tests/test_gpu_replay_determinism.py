"""Replays of a captured decode chain give the same bits every time (needs a GB300).

The decode attention kernel refills its shared-memory ring with tensor copies
while its warps read the previous tile with ldmatrix.  Those are two memory
proxies, and only a proxy fence orders them.  Without the fence, a copy
sometimes landed while a warp's last ldmatrix (V dims 112-127) was still
pending.  That needed the o_proj GEMV launched as a programmatic dependent,
its CTAs streaming weights beside attention's last wave.  Results then
changed from one replay to the next.

This test builds that situation.  A CUDA graph holds several copies of
[attention -> o_proj GEMV] over 8 layers.  Each (copy, layer) has its own
output and workspace, and all copies compute the same thing.  Every replay
must reproduce the first replay's attention outputs bit for bit.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

B, NH, NKV, HD = 8, 16, 8, 128     # the 0.6B shape with tp=2: 8 sequences, GQA group 2
CAP, CTX = 2176, 2049              # 2048 prompt keys + this step's key
HIDDEN, LAYERS, COPIES, REPLAYS = 1024, 8, 16, 100


def chain_mismatches(L, copies=COPIES, replays=REPLAYS, layers=LAYERS, history_ready=False):
    """Number of (replay, copy, layer) attention outputs that differ from replay 0."""
    g = torch.Generator(device="cuda").manual_seed(1234)
    bf = torch.bfloat16
    rnd = lambda *s, sc=1.0: (torch.randn(*s, device="cuda", generator=g) * sc).to(bf)  # noqa: E731
    kc = [rnd(B * CAP, NKV, HD, sc=0.5) for _ in range(layers)]
    vc = [rnd(B * CAP, NKV, HD) for _ in range(layers)]
    q = [rnd(B, NH, HD, sc=0.5) for _ in range(layers)]
    wo = [rnd(2, HIDDEN, NH * HD // 2, sc=0.02) for _ in range(layers)]   # row-split o_proj, tp=2
    cl = torch.full((B,), CTX, dtype=torch.int32, device="cuda")
    sb = torch.arange(B, dtype=torch.int32, device="cuda") * CAP
    ws_bytes = L.attention_decode_workspace_size(B, CAP, NH, HD)
    n = copies * layers
    ws = [torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda") for _ in range(n)]
    attn = [torch.empty(B, NH * HD, dtype=bf, device="cuda") for _ in range(n)]
    hout = [torch.empty(B, HIDDEN, dtype=bf, device="cuda") for _ in range(n)]

    def chain():
        for c in range(copies):
            for l in range(layers):
                i = c * layers + l
                L.attention_decode(q[l], kc[l], vc[l], cl, sb, CAP, NH, NKV, HD, HD ** -0.5, attn[i], ws[i],
                                   history_ready=history_ready)
                L.gemm(attn[i], wo[l], hout[i], HIDDEN, 2, L.QW_GEMM_ROW_REDUCE, L.QW_EPI_NONE)

    chain()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        chain()
    graph.replay()
    torch.cuda.synchronize()
    ref = [a.clone() for a in attn[:layers]]   # copy 0 of the first replay
    bad = 0
    for _ in range(replays):
        graph.replay()
        torch.cuda.synchronize()
        for i in range(n):
            if not torch.equal(attn[i], ref[i % layers]):
                bad += 1
    L.device_error()
    return bad


@pytest.mark.parametrize("history_ready", [False, True])
def test_decode_chain_replays_bit_identical(history_ready):
    """history_ready: the kernel before each attention is a GEMV that writes
    neither q nor the caches, so attention may stream its history early."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_transformer_forward_gb300 import build
    build.build()
    from qwen3_transformer_forward_gb300 import _lib as L
    L.load()
    assert chain_mismatches(L, history_ready=history_ready) == 0
