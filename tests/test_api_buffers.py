"""The binding checks every caller-provided buffer before a pointer crosses the C ABI.

The library receives bare device pointers and cannot see a tensor's size, dtype or
device: a wrong-shaped `out` would be written out of bounds on the GPU. These CPU
tests exercise the checks themselves (no launch, no GPU); the GPU test at the end
calls the real entry points with bad buffers and expects ValueError before any launch.
"""
import pytest
import torch

from paged_kv_cache_77_gb300 import api

CPU = torch.device("cpu")


def test_out_buffer_accepts_exact_shape_and_creates_when_absent():
    o = torch.empty((2, 3, 4), dtype=torch.float32)
    assert api.out_buffer(o, (2, 3, 4), torch.float32, CPU) is o
    ob = torch.empty((2, 3, 4), dtype=torch.bfloat16)
    assert api.out_buffer(ob, (2, 3, 4), torch.float32, CPU) is ob  # out's own dtype wins
    made = api.out_buffer(None, (2, 3, 4), torch.bfloat16, CPU)
    assert made.shape == (2, 3, 4) and made.dtype == torch.bfloat16


@pytest.mark.parametrize("bad", [
    torch.empty((2, 3, 5), dtype=torch.float32),            # wrong last dim
    torch.empty((2, 3, 4, 1), dtype=torch.float32),         # extra dim
    torch.empty((24,), dtype=torch.float32),                # flat, same numel
    torch.empty((2, 3, 4), dtype=torch.float16),            # unsupported dtype
    torch.empty((2, 3, 4), dtype=torch.int32),
    torch.empty((2, 4, 3), dtype=torch.float32).transpose(1, 2),  # non-contiguous
])
def test_out_buffer_rejects(bad):
    with pytest.raises(ValueError):
        api.out_buffer(bad, (2, 3, 4), torch.float32, CPU)


def test_out_buffer_rejects_other_device():
    meta = torch.empty((2, 3, 4), dtype=torch.float32, device="meta")
    with pytest.raises(ValueError, match="expected cpu"):
        api.out_buffer(meta, (2, 3, 4), torch.float32, CPU)


def test_out_dtype_must_be_supported_when_created():
    with pytest.raises(ValueError):
        api.out_buffer(None, (2, 3), torch.float16, CPU)


@pytest.mark.parametrize("bad", [
    torch.empty((2, 3), dtype=torch.bfloat16),
    torch.empty((2, 3), dtype=torch.float64),
    torch.empty((3, 2), dtype=torch.float32),
    torch.empty((2, 3, 1), dtype=torch.float32),
    torch.empty((3, 2), dtype=torch.float32).t(),
    torch.empty((2, 3), dtype=torch.float32, device="meta"),
])
def test_lse_buffer_rejects(bad):
    with pytest.raises(ValueError):
        api.lse_buffer(bad, (2, 3), CPU)


def test_lse_buffer_accepts_none_and_exact():
    assert api.lse_buffer(None, (2, 3), CPU) is None
    t = torch.empty((2, 3), dtype=torch.float32)
    assert api.lse_buffer(t, (2, 3), CPU) is t


def test_workspace_counts_bytes_not_elements():
    ws = torch.empty(100, dtype=torch.float32)  # 400 bytes
    got, nbytes = api.workspace_buffer(ws, 400, CPU)
    assert got is ws and nbytes == 400
    with pytest.raises(ValueError, match="needs 401"):
        api.workspace_buffer(ws, 401, CPU)
    with pytest.raises(ValueError):
        api.workspace_buffer(torch.empty((20, 20), dtype=torch.uint8).t(), 10, CPU)
    made, n = api.workspace_buffer(None, 1000, CPU)
    assert made.dtype == torch.uint8 and n >= 1000


def test_status_buffer():
    assert api.status_buffer(None, CPU) is None
    with pytest.raises(ValueError):
        api.status_buffer(torch.zeros(1, dtype=torch.int64), CPU)
    with pytest.raises(ValueError):
        api.status_buffer(torch.zeros(0, dtype=torch.int32), CPU)
    st = torch.zeros(1, dtype=torch.int32)
    assert api.status_buffer(st, CPU) is st


def test_inputs_must_be_cuda_tensors():
    # On a CPU-only machine every device call stops at its first input check.
    q = torch.zeros((1, 8, 128), dtype=torch.bfloat16)
    c = torch.zeros((2, 128, 8, 128), dtype=torch.bfloat16)
    t = torch.zeros((1, 2), dtype=torch.int32)
    lens = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        api.paged_attention_decode(q, c, c, t, lens, 0.1)
    with pytest.raises(ValueError, match="CUDA"):
        api.paged_attention_decode_static(q, c, c, t, lens, 0.1)


@pytest.mark.gpu
def test_entry_points_reject_bad_buffers_before_launch():
    dev = torch.device("cuda", torch.cuda.current_device())
    B, H, Hkv, d = 2, 8, 2, 128
    q = torch.zeros((B, H, d), dtype=torch.bfloat16, device=dev)
    c = torch.zeros((3, 128, Hkv, d), dtype=torch.bfloat16, device=dev)
    t = torch.zeros((B, 2), dtype=torch.int32, device=dev)
    lens = torch.zeros(B, dtype=torch.int32, device=dev)
    cases = [
        dict(out=torch.empty((B, H, d - 1), dtype=torch.float32, device=dev)),
        dict(out=torch.empty((B * H * d,), dtype=torch.float32, device=dev)),
        dict(out=torch.empty((B, H, d), dtype=torch.float16, device=dev)),
        dict(out=torch.empty((B, H, d), dtype=torch.float32)),  # host tensor
        dict(lse=torch.empty((B, H + 1), dtype=torch.float32, device=dev)),
        dict(lse=torch.empty((B, H), dtype=torch.bfloat16, device=dev)),
        dict(workspace=torch.empty(16, dtype=torch.uint8, device=dev)),
        dict(dev_status=torch.zeros(1, dtype=torch.int64, device=dev)),
    ]
    for kw in cases:
        with pytest.raises(ValueError):
            api.paged_attention_decode(q, c, c, t, lens, 0.1, **kw)
    with pytest.raises(ValueError):
        api.paged_attention_decode(q, c[:, :, :, :64].contiguous(), c, t, lens, 0.1)
    with pytest.raises(ValueError):
        api.paged_attention_decode(q, c, c, t[:1], lens, 0.1)
    qn = torch.zeros((B, H, 512), dtype=torch.bfloat16, device=dev)
    qr = torch.zeros((B, H, 64), dtype=torch.bfloat16, device=dev)
    cn = torch.zeros((3, 128, 1, 512), dtype=torch.bfloat16, device=dev)
    cr = torch.zeros((3, 128, 1, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        api.mla_paged_decode(qn, qr, cn, cr, t, lens, 0.1,
                             out=torch.empty((B, H, 256), dtype=torch.float32, device=dev))
    with pytest.raises(ValueError):
        api.mla_paged_decode(qn, qr, cn, cr, t, lens, 0.1,
                             lse=torch.empty((B,), dtype=torch.float32, device=dev))
    cu = torch.tensor([1, 2], dtype=torch.int32, device=dev)
    with pytest.raises(ValueError):
        api.paged_attention_prefill(q, cu, c, c, t, lens, 0.1,
                                    out=torch.empty((B, H, d), dtype=torch.float32,
                                                    device=dev).transpose(0, 1))
    torch.cuda.synchronize()
