"""Past-the-end canaries on every output buffer the kernels write.

Each output is the leading part of a larger allocation whose remainder (a
guard of at least one row, or 64 extra elements after a column-major scale
buffer) holds a sentinel byte pattern.  After the call the guard must be
untouched, and so must the entries between `rows` and the leading dimension
of a column-major buffer.  The bulk-store kernels move whole rows with TMA
copies, so this catches a row written one past the end or a copy of the
wrong length.  Shapes are ragged (T not a multiple of the tokens per CTA,
R larger than T*k, H not a multiple of 512, G not a multiple of 4) and every
pos table names row R - 1.
"""
import pytest
import torch

from moe_routing_precision_gb300 import ops, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FILL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_routing_precision_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    assert ops.device_status() == 0
    yield
    assert ops.device_status() == 0


class Guarded:
    """A `shape` buffer of `dtype` at the front of an allocation with `extra`
    more elements (default: one more row) all set to the sentinel byte."""

    def __init__(self, shape, dtype, extra=None):
        n = 1
        for s in shape:
            n *= s
        row = n // shape[0] if shape[0] else n
        extra = row if extra is None else extra
        esz = torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full(((n + extra) * esz,), FILL, dtype=torch.uint8, device=DEV)
        self.n_bytes = n * esz
        self.view = self.raw[:self.n_bytes].view(dtype).view(*shape)

    def guard_intact(self):
        tail = self.raw[self.n_bytes:]
        return bool((tail == FILL).all())


def _pos_with_last_row(T, k, R, seed):
    """pos [T, k]: distinct rows of [0, R) that include R - 1."""
    assert R >= T * k
    g = torch.Generator().manual_seed(seed)
    rows = torch.randperm(R, generator=g)[:T * k]
    if (rows == R - 1).sum() == 0:
        rows[seed % rows.numel()] = R - 1
    return rows.to(torch.int32).view(T, k).to(DEV)


EXPAND_SHAPES = [(1, 512, 1, 3), (3, 7168, 8, 29), (33, 1024, 2, 70), (5, 384, 3, 16),
                 (7, 896, 4, 29), (4, 20480, 2, 9)]   # bulk, bulk, bulk, rows (G=3), rows (G=7), tile


@pytest.mark.parametrize("T,H,k,R", EXPAND_SHAPES)
def test_expand_fp8_guards(T, H, k, R):
    x = workloads.random_small(T, 16, k, H, seed=T + H)["x"].to(DEV)
    pos = _pos_with_last_row(T, k, R, T + k)
    q = Guarded((R, H), torch.uint8)
    sf = Guarded((R, H // 128), torch.float32)
    ops.expand_cast_fp8(x, pos, R, out=q.view, out_sf=sf.view)
    assert ops.device_status() == 0
    assert q.guard_intact() and sf.guard_intact()
    assert int((q.view[R - 1] == FILL).sum()) < H          # the last row was written


@pytest.mark.parametrize("T,H,k,align", [(9, 1024, 3, 16), (37, 7168, 8, 128), (5, 384, 2, 8)])
def test_expand_fp8_padded_guards(T, H, k, align):
    E = 16
    x = workloads.random_small(T, E, k, H, seed=T)["x"].to(DEV)
    idx = torch.rand(T, E, generator=torch.Generator().manual_seed(T)).argsort(1)[:, :k]
    _, _, pos, src = ops.route_map_aligned(idx.to(torch.int32).to(DEV).contiguous(), E, align)
    R = src.shape[0]
    q = Guarded((R, H), torch.uint8)
    sf = Guarded((R, H // 128), torch.float32)
    ops.expand_cast_fp8_padded(x, pos, src, out=q.view, out_sf=sf.view)
    assert ops.device_status() == 0
    assert q.guard_intact() and sf.guard_intact()


def _colmajor_sf(rows, G, flags, like_extra=64):
    ld = (rows + 3) // 4 * 4 + 4          # 4 spare columns between rows and ld
    if flags & ops.SF_UE8M0:
        buf = Guarded(((G + 3) // 4, ld, 4), torch.uint8, extra=like_extra)
    else:
        buf = Guarded((G, ld), torch.float32, extra=like_extra)
    return buf, ld


def _between_rows_and_ld_intact(buf, rows, flags):
    v = buf.view.view(torch.uint8) if flags & ops.SF_UE8M0 else buf.view.view(torch.int32)
    if flags & ops.SF_UE8M0:
        return bool((v[:, rows:, :] == FILL).all())
    return bool((v[:, rows:] == int.from_bytes(bytes([FILL] * 4), "little", signed=True)).all())


@pytest.mark.parametrize("flags", [ops.SF_COLMAJOR, ops.SF_COLMAJOR | ops.SF_POW2,
                                   ops.SF_COLMAJOR | ops.SF_POW2 | ops.SF_UE8M0,
                                   ops.SF_POW2 | ops.SF_UE8M0])
@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("T,H,k,R", [(3, 7168, 8, 29), (5, 640, 2, 13)])
def test_expand_fp8_ex_guards(flags, staged, T, H, k, R):
    x = workloads.random_small(T, 16, k, H, seed=T + 7)["x"].to(DEV)
    pos = _pos_with_last_row(T, k, R, T + 3)
    src = torch.full((R,), -1, dtype=torch.int32)
    p = pos.cpu().flatten()
    src[p.long()] = torch.arange(T * k, dtype=torch.int32)
    src = src.to(DEV)
    G = H // 128
    q = Guarded((R, H), torch.uint8)
    if flags & ops.SF_COLMAJOR:
        sf, ld = _colmajor_sf(R, G, flags)
    else:
        sf, ld = Guarded((R, G), torch.uint8), None
    ops.expand_cast_fp8_ex(x, pos, R, sorted_src=src, sf_flags=flags, sf_ld=ld, out=q.view,
                           out_sf=sf.view, workspace=True if staged else None)
    assert ops.device_status() == 0
    assert q.guard_intact() and sf.guard_intact()
    if flags & ops.SF_COLMAJOR:
        assert _between_rows_and_ld_intact(sf, R, flags)


@pytest.mark.parametrize("group", [16, 32, 128])
@pytest.mark.parametrize("T,H,k,R", [(3, 7168, 8, 27), (5, 96, 2, 11), (9, 1024, 4, 40)])
def test_expand_fp4_guards(group, T, H, k, R):
    if H % group:
        pytest.skip("H not a multiple of the group")
    x = workloads.random_small(T, 16, k, H, seed=T + group)["x"].to(DEV)
    pos = _pos_with_last_row(T, k, R, T + group)
    q = Guarded((R, H // 2), torch.uint8)
    sf = Guarded((R, H // group), torch.float32)
    ops.expand_cast_fp4(x, pos, R, group=group, out=q.view, out_sf=sf.view)
    assert ops.device_status() == 0
    assert q.guard_intact() and sf.guard_intact()


@pytest.mark.parametrize("M,N", [(1, 128), (37, 2048), (1001, 384)])
def test_swiglu_guards(M, N):
    g = torch.Generator().manual_seed(M + N)
    x = torch.randn(M, 2 * N, generator=g).to(torch.bfloat16).to(DEV)
    q = Guarded((M, N), torch.uint8)
    sf = Guarded((M, N // 128), torch.float32)
    ops.swiglu_cast_fp8(x, out=q.view, out_sf=sf.view)
    q4 = Guarded((M, N // 2), torch.uint8)
    sf4 = Guarded((M, N // 32), torch.float32)
    ops.swiglu_cast_fp4(x, group=32, out=q4.view, out_sf=sf4.view)
    assert ops.device_status() == 0
    assert all(b.guard_intact() for b in (q, sf, q4, sf4))


@pytest.mark.parametrize("T,H,k", [(3, 7168, 8), (33, 136, 3), (1, 8, 1)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_combine_guards(T, H, k, dtype):
    R = T * k + 2
    g = torch.Generator().manual_seed(T * H)
    y = torch.randn(R, H, generator=g).to(torch.bfloat16).to(DEV)
    w = torch.rand(T, k, generator=g).to(DEV)
    pos = _pos_with_last_row(T, k, R, T)
    out = Guarded((T, H), dtype)
    ops.combine(y, w, pos, dtype, out=out.view)
    assert ops.device_status() == 0
    assert out.guard_intact()
