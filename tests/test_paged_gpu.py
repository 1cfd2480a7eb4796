"""GPU parity of decode against a paged, variable-length KV cache
(attn_fwd_paged_decode) with the oracle's paged_decode_attention, on the
same 16-bit pages and block tables.

Caches are drawn contiguous with the seeded generator, then laid out in a
pool of pages in a seeded random order (unused rows of a page hold
garbage, which must never be read). Cases span lengths that end inside a
page, a zero length, page sizes 1 to 256, grouped-query heads, d = 64 and
128, bf16 and fp16, automatic and fixed split counts, and the 32 x 12-head,
16K-key decode workload in pages, checked on sampled rows."""

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_attn_gb300 import _lib
from exact_io_aware_attn_gb300.inputs import BF16, F16, make_qkv
from parity_helpers import UNIT_ROUNDOFF, oracle_scale

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_device):
    from exact_io_aware_attn_gb300 import build
    build.build()
    yield


def make_paged(B, h_q, h_kv, lens, d, dtype, page_size, seed, spare=5):
    """q [B, h_q, d]; pools [num_pages, h_kv, page_size, d]; table; lens."""
    T = max(1, max(lens))
    q, k, v = make_qkv(B, h_q, 1, T, d, dtype, seed=seed, h_kv=h_kv)
    q = q[:, :, 0]
    max_pages = -(-T // page_size)
    num_pages = B * max_pages + spare
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages)
    shape = (num_pages, h_kv, page_size, d)
    if num_pages * h_kv * page_size * d <= (1 << 24):
        # rows no sequence owns hold large garbage: reading one shows up
        gen = torch.Generator().manual_seed(seed + 7)
        kp = (torch.randn(shape, generator=gen) * 30.0).to(k.dtype)
        vp = (torch.randn(shape, generator=gen) * 30.0).to(v.dtype)
    else:
        kp = torch.zeros(shape, dtype=k.dtype)
        vp = torch.zeros(shape, dtype=v.dtype)
    table = np.full((B, max_pages), int(perm[-1]), dtype=np.int32)
    n = 0
    for b in range(B):
        for j in range(-(-lens[b] // page_size)):
            pg = int(perm[n])
            n += 1
            table[b, j] = pg
            r0, r1 = j * page_size, min((j + 1) * page_size, lens[b])
            kp[pg, :, : r1 - r0] = k[b, :, r0:r1]
            vp[pg, :, : r1 - r0] = v[b, :, r0:r1]
    return q, kp, vp, torch.from_numpy(table), torch.tensor(lens, dtype=torch.int32)


def gpu_paged(q, kp, vp, table, lens, num_splits=0, check_status=True):
    dev = torch.device("cuda:0")
    o = torch.full(q.shape, float("nan"), dtype=q.dtype, device=dev)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    _lib.attn_fwd_paged_decode(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), lens.to(dev),
                               out=o, lse=lse, num_splits=num_splits)
    torch.cuda.synchronize()
    if check_status:
        st, word = _lib.get_device_error()
        assert st == _lib.ATTN_OK, f"device status {st} word {word:#x}"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_paged(q, kp, vp, table, lens, rows=None):
    s = oracle_scale(q.shape[-1] ** -0.5)
    tn, ln = table.numpy(), lens.numpy()
    if rows is not None:
        # only the sampled sequences, with only the pages they use
        q, tn, ln = q[rows], tn[rows], ln[rows]
        used = np.unique(tn)
        remap = {int(p): i for i, p in enumerate(used)}
        tn = np.vectorize(lambda p: remap[int(p)])(tn).astype(np.int32)
        kp, vp = kp[torch.from_numpy(used).long()], vp[torch.from_numpy(used).long()]
    qn, kn, vn = q.double().numpy(), kp.double().numpy(), vp.double().numpy()
    o, lse = oracle.paged_decode_attention(qn, kn, vn, tn, ln, scale=s)
    o_abs, _ = oracle.paged_decode_attention(qn, kn, np.abs(vn), tn, ln, scale=s)
    return o, lse, o_abs


def compare_paged(o, lse, ref, dtype, what):
    o_ref, lse_ref, o_abs = ref
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf lse pattern differs"
    assert np.all(o[empty] == 0), f"{what}: zero-length rows must give o = 0"
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    full = ~empty
    err_l = np.abs(lse[full] - lse_ref[full])
    assert err_l.size == 0 or err_l.max() <= 1e-3, f"{what}: max|dlse| = {err_l.max():.3e}"
    u = UNIT_ROUNDOFF[dtype]
    err = np.abs(o - o_ref)
    bound = 1.25 * u * (o_abs + np.abs(o_ref)) + 1e-4
    worst = np.argmax(err / bound)
    assert (err <= bound).all(), (f"{what}: element {np.unravel_index(worst, o.shape)} off by "
                                  f"{err.flat[worst]:.3e} (bound {bound.flat[worst]:.3e})")
    assert err.max() <= 2e-2


CASES = [
    # B, h_q, h_kv, lens, d, dtype, page_size, splits
    (3, 8, 2, [1000, 1, 517], 64, BF16, 16, 0),
    (3, 8, 2, [1000, 1, 517], 64, BF16, 16, 7),
    (3, 4, 4, [320, 3, 0], 128, F16, 64, 0),        # a zero-length sequence
    (2, 6, 3, [77, 130], 64, F16, 1, 5),            # one row per page
    (2, 2, 1, [16384, 9000], 64, BF16, 256, 0),     # long, group 2
    (4, 12, 12, [33, 64, 65, 200], 128, BF16, 32, 0),
    (1, 1, 1, [5], 64, BF16, 64, 16),               # more partitions than keys
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(str(x) for x in c[:3]) + f"_ps{c[6]}_s{c[7]}_d{c[4]}")
def test_paged_decode_parity(case):
    B, hq, hkv, lens, d, dt, ps, splits = case
    q, kp, vp, table, ln = make_paged(B, hq, hkv, lens, d, dt, ps, seed=41)
    o, lse = gpu_paged(q, kp, vp, table, ln, splits)
    compare_paged(o, lse, oracle_paged(q, kp, vp, table, ln), dt, f"paged {case}")


def test_paged_equals_contiguous_decode():
    """With every page in order and full lengths, the paged path reads the
    same keys as the contiguous decode: both within the gate of the oracle
    and of each other."""
    B, h, T, d, ps = 2, 4, 700, 64, 16
    q, k, v = make_qkv(B, h, 1, T, d, BF16, seed=42)
    max_pages = -(-T // ps)
    kp = torch.zeros(B * max_pages, h, ps, d, dtype=k.dtype)
    vp = torch.zeros_like(kp)
    for b in range(B):
        for j in range(max_pages):
            r1 = min((j + 1) * ps, T)
            kp[b * max_pages + j, :, : r1 - j * ps] = k[b, :, j * ps:r1]
            vp[b * max_pages + j, :, : r1 - j * ps] = v[b, :, j * ps:r1]
    table = torch.arange(B * max_pages, dtype=torch.int32).reshape(B, max_pages)
    lens = torch.full((B,), T, dtype=torch.int32)
    o_p, l_p = gpu_paged(q[:, :, 0], kp, vp, table, lens, 8)
    o_c, l_c = _lib.attn_fwd(q.cuda(), k.cuda(), v.cuda(), num_splits=8)
    assert np.abs(o_p - o_c.double().cpu().numpy()[:, :, 0]).max() <= 2e-2
    assert np.abs(l_p - l_c.double().cpu().numpy()[:, :, 0]).max() <= 1e-3


def test_paged_bad_table_entry_is_reported_not_read():
    q, kp, vp, table, ln = make_paged(2, 4, 2, [100, 50], 64, BF16, 16, seed=43)
    bad = table.clone()
    bad[0, 2] = kp.shape[0] + 7     # outside the pool
    bad[1, 0] = -3
    gpu_paged(q, kp, vp, bad, ln, check_status=False)
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_ERR_INVALID_ARG
    assert (word >> 8) & 0xff == 7          # the paged split kernel
    # reading cleared it; a valid call afterwards is clean and correct
    o, lse = gpu_paged(q, kp, vp, table, ln)
    compare_paged(o, lse, oracle_paged(q, kp, vp, table, ln), BF16, "after a bad table")


def test_paged_full_size_sampled_rows():
    """The 32 x 12-head, 16K-key bf16 decode workload laid out in 64-row
    pages in random order, one call; four whole sequences (48 rows) checked
    against the oracle run on those sequences alone."""
    B, h, T, d, ps = 32, 12, 16384, 64, 64
    lens = [T] * B
    q, kp, vp, table, ln = make_paged(B, h, h, lens, d, BF16, ps, seed=44, spare=0)
    o, lse = gpu_paged(q, kp, vp, table, ln)
    rows = np.array([0, 7, 13, 31])
    ref = oracle_paged(q, kp, vp, table, ln, rows=rows)
    compare_paged(o[rows], lse[rows], ref, BF16, "paged full size")


def test_paged_kernel_name_and_workspace():
    q, kp, vp, table, ln = make_paged(2, 4, 2, [100, 50], 128, F16, 16, seed=45)
    nbytes = _lib.paged_workspace_bytes(2, 4, 2, 128, 16, table.shape[1], 6)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    _lib.attn_fwd_paged_decode(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), ln.cuda(),
                               num_splits=6, workspace=ws)
    torch.cuda.synchronize()
    assert _lib.last_kernel_name() == "decode_paged_split_d128_f16+decode_combine"
    with pytest.raises(_lib.AttnError) as e:
        _lib.attn_fwd_paged_decode(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), ln.cuda(),
                                   num_splits=6, workspace=ws[:64])
    assert e.value.status == _lib.ATTN_ERR_WORKSPACE


TC_CASES = [
    # B, h_q, h_kv, lens, d, dtype, page_size, splits -- groups >= 4 with pages
    # of >= 8 rows: the tensor-core path (K/V tiles gathered through the table)
    (3, 8, 2, [1000, 1, 517], 64, BF16, 16, 0),
    (2, 16, 2, [4096, 3000], 128, BF16, 128, 0),
    (2, 16, 4, [300, 700], 64, F16, 8, 5),          # 8-row pages: 16 boxes per tile
    (3, 8, 1, [320, 3, 0], 128, BF16, 64, 0),       # a zero-length sequence, group 8
    (2, 12, 3, [2000, 129], 128, F16, 256, 1),      # one partition: no workspace
    (1, 32, 2, [16384], 64, BF16, 64, 64),          # group 16, the most partitions
    # one key/value head at d = 64: the two heads of a unit come from
    # different sequences (different lengths), the last unit has one head
    (3, 4, 1, [1000, 7, 517], 64, BF16, 16, 0),
    (3, 4, 1, [300, 0, 50], 64, BF16, 16, 1),       # length 0, one partition: o = 0
    # the same with 64- and 256-row pages: two heads per unit (head pairs),
    # each tile's table entries staged in shared memory
    (3, 4, 1, [1000, 7, 517], 64, BF16, 64, 0),
    (3, 4, 1, [300, 0, 50], 64, F16, 64, 1),
    (3, 4, 1, [2500, 130, 1], 64, BF16, 256, 3),
    (2, 16, 4, [5000, 4999], 64, BF16, 128, 0),     # same sequence in both heads
    (4, 8, 1, [0, 2000, 64, 900], 64, F16, 8, 0),   # length 0 in a unit's first head
    # pages of >= 64 rows at d = 64: two heads per unit, each with its own
    # page lookups (pipelined one key tile ahead)
    (3, 4, 1, [1000, 7, 517], 64, BF16, 64, 0),
    (4, 8, 1, [0, 2000, 64, 900], 64, F16, 128, 0),
    (3, 4, 1, [300, 0, 50], 64, BF16, 256, 1),      # length 0, one partition: o = 0
    (2, 8, 2, [4000, 3000], 64, BF16, 64, 3),
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "x".join(str(x) for x in c[:3]) + f"_ps{c[6]}_s{c[7]}_d{c[4]}")
def test_paged_decode_tensor_core_path(case):
    B, hq, hkv, lens, d, dt, ps, splits = case
    q, kp, vp, table, ln = make_paged(B, hq, hkv, lens, d, dt, ps, seed=46)
    o, lse = gpu_paged(q, kp, vp, table, ln, splits)
    assert _lib.last_kernel_name().startswith("prefill_paged_tcgen05")
    compare_paged(o, lse, oracle_paged(q, kp, vp, table, ln), dt, f"paged tc {case}")


@pytest.mark.parametrize("ps", [16, 64])
def test_paged_tensor_core_bad_table_entry_is_reported(ps):
    # 16-row pages: one head per unit, the entry read per box; 64-row pages:
    # head pairs, the entry read while the unit's entries are staged
    q, kp, vp, table, ln = make_paged(2, 8, 2, [300, 200], 64, BF16, ps, seed=47)
    bad = table.clone()
    bad[1, 1] = kp.shape[0] + 3
    gpu_paged(q, kp, vp, bad, ln, check_status=False)
    st, word = _lib.get_device_error()
    assert st == _lib.ATTN_ERR_INVALID_ARG
    assert (word >> 8) & 0xff == 1          # the prefill kernel's producer
    o, lse = gpu_paged(q, kp, vp, table, ln)
    compare_paged(o, lse, oracle_paged(q, kp, vp, table, ln), BF16, "tc after a bad table")
