"""Host-side checks of the C ABI: the library builds, loads, exports every
function that include/fa.h declares, and rejects bad arguments before touching
the GPU (these calls return from validation without any CUDA call)."""
import ctypes
import os

import pytest
import torch

import exact_attention_30_gb300 as fa
from exact_attention_30_gb300 import build as fa_build


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.library_path()):
        fa_build.build()
    return fa.load_library()


def test_header_declares_expected_entry_points():
    names = fa.header_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_check_device_status",
              "fa_status_string", "fa_version", "fa_debug_timeout_probe"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in fa.header_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert fa.fa_status_string(fa.FA_OK) == "FA_OK"
    for code in (fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED, fa.FA_ERR_CUDA, fa.FA_ERR_TIMEOUT):
        assert fa.fa_status_string(code).startswith("FA_ERR_")
    assert fa.fa_version() >= 100


def test_workspace_size_is_host_only(lib):
    n = fa.fa_bwd_workspace_bytes(2, 16, 4096, 128)
    # dQ accumulator (fp32) + two fp32 row statistics, rows padded to 128
    assert n >= 2 * 16 * 4096 * 128 * 4 + 2 * 2 * 16 * 4096 * 4
    assert n % 256 == 0
    assert lib.fa_bwd_workspace_bytes(0, 1, 1, 64, fa.FA_BF16) == 0
    assert lib.fa_bwd_workspace_bytes(1, 1, 1, 96, fa.FA_BF16) == 0  # unsupported d
    assert lib.fa_bwd_workspace_bytes(1, 1, 1000, 64, fa.FA_F32) >= 4000


def test_packed_batch_workspace_holds_the_schedule(lib):
    # the main kernel's schedule follows the per-row buffers: the unit counter
    # and total, then the sequence order and the B + 1 unit prefix sums
    H, total, max_len, d = 2, 4096, 2048, 64
    one = lib.fa_bwd_varlen_workspace_bytes(2, H, total, max_len, d, fa.FA_BF16)
    many = lib.fa_bwd_varlen_workspace_bytes(2000, H, total, max_len, d, fa.FA_BF16)
    assert one > 0 and one % 256 == 0 and many % 256 == 0
    # two ints more per sequence, less the 256-byte padding of the small schedule
    assert many - one >= 4 * 2 * (2000 - 2) - 256
    # fixed length: the counter and the total only (one 256-byte block)
    assert fa.fa_bwd_workspace_bytes(1, 1, 128, 64) >= 128 * 64 * 4 + 2 * 128 * 4 + 256


FAKE = 0x10000  # an aligned non-null value: never dereferenced, validation fails first


@pytest.mark.parametrize("args,code", [
    ((0, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 64, 0.125, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 16, 64, 0.125, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 0, 64, 0.125, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 64, 0.0, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 64, float("nan"), fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 96, 0.125, fa.FA_BF16), fa.FA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 256, 0.125, fa.FA_F32), fa.FA_ERR_UNSUPPORTED),
    ((FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 64, 0.125, fa.FA_BF16), fa.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 64, 0.125, 7), fa.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 70000, 1, 16, 64, 0.125, fa.FA_BF16), fa.FA_ERR_UNSUPPORTED),
])
def test_fwd_rejects_bad_arguments_before_launch(lib, args, code):
    assert lib.fa_fwd(*args, None) == code


def test_bwd_rejects_small_workspace_and_nulls(lib):
    ws = fa.fa_bwd_workspace_bytes(1, 2, 300, 64)
    ptrs = [FAKE] * 10
    assert lib.fa_bwd(*ptrs, ws - 1, 1, 2, 300, 64, 0.125, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    bad = list(ptrs)
    bad[6] = 0  # dQ
    assert lib.fa_bwd(*bad, ws, 1, 2, 300, 64, 0.125, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    bad = list(ptrs)
    bad[9] = FAKE + 16  # workspace not 256-byte aligned
    assert lib.fa_bwd(*bad, ws, 1, 2, 300, 64, 0.125, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG


def test_python_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fa_fwd(q, q, q)


def test_softmax_rows_rejects_bad_arguments_before_launch(lib):
    assert lib.fa_softmax_rows(0, FAKE, 4, 16, 1.0, fa.FA_F32, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_softmax_rows(FAKE, FAKE, 0, 16, 1.0, fa.FA_F32, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_softmax_rows(FAKE, FAKE, 4, 16, 0.0, fa.FA_F32, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_softmax_rows(FAKE + 1, FAKE, 4, 16, 1.0, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_softmax_rows(FAKE, FAKE, 4, 32769, 1.0, fa.FA_F32, None) == fa.FA_ERR_UNSUPPORTED


def test_decode_rejects_bad_arguments_before_launch(lib):
    def call(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, ws=FAKE, ws_bytes=1 << 30, B=1, H=2, nq=1,
             nk=100, d=128, scale=0.088, dt=fa.FA_BF16):
        return lib.fa_decode(q, k, v, o, lse, ws, ws_bytes, B, H, nq, nk, d, scale, dt, None)
    assert call(q=0) == fa.FA_ERR_INVALID_ARG
    assert call(ws=0) == fa.FA_ERR_INVALID_ARG
    assert call(nk=0) == fa.FA_ERR_INVALID_ARG
    assert call(nq=0) == fa.FA_ERR_INVALID_ARG
    assert call(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert call(nq=17) == fa.FA_ERR_UNSUPPORTED
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(dt=fa.FA_F32) == fa.FA_ERR_UNSUPPORTED
    assert call(B=300, H=300) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_decode_workspace_bytes(1, 1, 17, 100, 128, fa.FA_BF16) == 0


def _plan_cost(BH, nk, slots, s, tile):
    kps = (-(-nk // s) + tile - 1) // tile * tile
    return -(-BH * s // slots) * (kps + 128), kps


@pytest.mark.parametrize("B,H,nq,nk,slots", [
    (8, 32, 1, 32768, 304), (1, 1, 1, 1, 304), (1, 1, 4, 1000, 304), (2, 3, 8, 70000, 456),
    (64, 32, 1, 4096, 304), (1, 8, 2, 131072, 608), (4, 4, 1, 100, 3)])
def test_decode_plan_on_the_host(lib, B, H, nq, nk, slots):
    """The split plan covers every key with non-empty whole-tile ranges (64-key
    tiles for one query per head, 128-key tensor-core tiles for more) and
    minimises waves x (keys per split + 128) over all admissible split counts."""
    tile = 64 if nq == 1 else 128
    s, kps = fa.fa_decode_plan(B, H, nq, nk, 128, resident_ctas=slots)
    assert kps % tile == 0 and 1 <= s <= 256
    assert s * kps >= nk and (s - 1) * kps < nk  # covers all keys, no empty range
    best = min(_plan_cost(B * H, nk, slots, t, tile)[0] for t in range(1, min(256, -(-nk // tile)) + 1)
               if -(-nk // _plan_cost(B * H, nk, slots, t, tile)[1]) == t)
    assert _plan_cost(B * H, nk, slots, s, tile)[0] == best


def _tail_makespan(units, slots, n_full, n_tail, splits):
    """Waves of whole-unit time: full waves, then the tail at 1/splits each
    (every tail range runs in the same wave when n_tail * splits <= slots)."""
    assert n_full % slots == 0 and n_tail * splits <= slots
    return n_full // slots + (1.0 / splits if n_tail else 0.0)


@pytest.mark.parametrize("B,H,N,d,slots", [
    (2, 16, 4096, 128, 152), (1, 32, 16384, 128, 152), (4, 16, 1024, 64, 152),
    (1, 10, 4096, 128, 152), (1, 10, 4000, 64, 152), (1, 4, 4096, 128, 152),
    (1, 200, 1024, 128, 152), (1, 200, 256, 128, 152), (3, 7, 777, 64, 148), (1, 1, 1, 128, 152),
    (2, 16, 4096, 64, 152), (1, 16, 16384, 64, 152), (1, 2, 20000, 64, 152)])
def test_forward_tail_split_plan_on_the_host(lib, B, H, N, d, slots):
    """The forward's tail split covers every unit once, splits only the last,
    partly filled wave (never with fewer than four key tiles per range, at
    most four ranges, all of them in one wave) and never lengthens the
    schedule; causal and fp32 problems are not split."""
    units = B * H * -(-N // 256)
    n_kv = -(-N // 128)
    nf, nt, sp = fa.fa_fwd_plan(B, H, N, d, resident_ctas=slots)
    assert nf + nt == units and sp >= 1 and (sp == 1) == (nt == 0)
    # d = 64 problems whose four-tile grid (one CTA per 512 rows) fills at
    # least 3/4 of the resident CTAs run unsplit on that kernel
    if d == 64 and 4 * B * H * -(-N // 512) >= 3 * slots:
        assert (nf, nt, sp) == (units, 0, 1)
    elif sp > 1:
        assert nt == units % slots and units >= slots
        assert 2 <= sp <= 4 and n_kv // sp >= 4 and nt * sp <= slots
        assert sp == min(slots // nt, 4, n_kv // 4)
        whole = -(-units // slots)
        assert _tail_makespan(units, slots, nf, nt, sp) < whole
    else:
        rem = units % slots
        assert rem == 0 or units < slots or min(slots // rem, 4, n_kv // 4) < 2
    assert fa.fa_fwd_plan(B, H, N, d, causal=True, resident_ctas=slots) == (units, 0, 1)
    assert fa.fa_fwd_plan(B, H, N, d, dtype=torch.float32, resident_ctas=slots) == (units, 0, 1)


def test_forward_workspace_entry_points_without_a_gpu(lib):
    # no device: nothing is split, so no scratch is asked for
    assert lib.fa_fwd_workspace_bytes(2, 16, 4096, 128, 0, fa.FA_BF16) == 0
    assert lib.fa_fwd_workspace_bytes(2, 16, 4096, 96, 0, fa.FA_BF16) == 0
    assert lib.fa_fwd_workspace_bytes(2, 16, 4096, 128, 4, fa.FA_BF16) == 0
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE)
    assert lib.fa_fwd_ws(*ok, None, 0, 1, 2, 64, 64, 0.125, 4, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_ws(*ok, None, 0, 0, 2, 64, 64, 0.125, 0, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    nf = ctypes.c_int()
    assert lib.fa_fwd_plan(1, 1, 64, 64, 0, fa.FA_BF16, -1, ctypes.byref(nf), ctypes.byref(nf),
                           ctypes.byref(nf)) == fa.FA_ERR_INVALID_ARG


def test_ex_and_varlen_entry_points_reject_bad_arguments_before_launch(lib):
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE)
    # unknown flags
    assert lib.fa_fwd_ex(*ok, 1, 2, 64, 64, 0.125, 4, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    ws = fa.fa_bwd_workspace_bytes(1, 2, 64, 64)
    assert lib.fa_bwd_ex(*([FAKE] * 10), ws, 1, 2, 64, 64, 0.125, 1 << 12, fa.FA_BF16,
                         None) == fa.FA_ERR_INVALID_ARG

    def fwd_v(cu=FAKE, B=2, H=3, total=100, maxlen=60, d=64, scale=0.125, flags=0, dt=fa.FA_BF16):
        return lib.fa_fwd_varlen(*ok, cu, B, H, total, maxlen, d, scale, flags, dt, None)
    assert fwd_v(cu=0) == fa.FA_ERR_INVALID_ARG           # no offsets
    assert fwd_v(cu=FAKE + 2) == fa.FA_ERR_INVALID_ARG    # misaligned offsets
    assert fwd_v(maxlen=101) == fa.FA_ERR_INVALID_ARG     # longer than the batch
    assert fwd_v(total=0) == fa.FA_ERR_INVALID_ARG
    assert fwd_v(flags=2) == fa.FA_ERR_INVALID_ARG
    assert fwd_v(d=96) == fa.FA_ERR_UNSUPPORTED
    assert fwd_v(B=70000) == fa.FA_ERR_UNSUPPORTED
    # workspace sizes: host only, grow with the packed rows, 0 on bad sizes
    n1 = fa.fa_bwd_varlen_workspace_bytes(2, 3, 100, 60, 64)
    n2 = fa.fa_bwd_varlen_workspace_bytes(2, 3, 1000, 600, 64)
    assert 0 < n1 < n2 and n1 % 256 == 0
    assert lib.fa_bwd_varlen_workspace_bytes(2, 3, 100, 101, 64, fa.FA_BF16) == 0
    assert lib.fa_bwd_varlen(*([FAKE] * 11), n1 - 1, 2, 3, 100, 60, 64, 0.125, 0, fa.FA_BF16,
                             None) == fa.FA_ERR_INVALID_ARG  # workspace too small


def test_python_binding_checks_varlen_arguments():
    import torch
    q = torch.zeros(10, 2, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 10], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fa_fwd_varlen(q, q, q, cu, 10)


@pytest.mark.parametrize("B,H,N,d,slots", [
    (2, 16, 4096, 128, 152), (4, 16, 1024, 64, 152), (1, 16, 4096, 128, 152), (1, 10, 2000, 128, 152),
    (1, 32, 16384, 128, 152), (1, 1, 1, 64, 152), (1, 5, 8192, 64, 148), (3, 7, 700, 128, 152)])
def test_backward_tail_split_plan_on_the_host(lib, B, H, N, d, slots):
    """The backward's tail split covers every (head, key tile) unit once, splits
    only a last wave that fills at most half the SMs (ranges of at least four
    query tiles, at most four ranges, all in that wave) and shortens the
    schedule; causal and fp32 problems are never split."""
    n_q = -(-N // 128)
    units = B * H * n_q
    nf, nt, sp = fa.fa_bwd_plan(B, H, N, d, resident_ctas=slots)
    assert nf + nt == units and sp >= 1 and (sp == 1) == (nt == 0)
    if sp > 1:
        assert nt == units % slots and units >= slots
        assert 2 <= sp <= 4 and n_q // sp >= 4 and nt * sp <= slots
        assert sp == min(slots // nt, 4, n_q // 4)
        assert nf // slots + 1.0 / sp < -(-units // slots)
    else:
        rem = units % slots
        assert rem == 0 or units < slots or min(slots // rem, 4, n_q // 4) < 2
    assert fa.fa_bwd_plan(B, H, N, d, causal=True, resident_ctas=slots) == (units, 0, 1)
    assert fa.fa_bwd_plan(B, H, N, d, dtype=torch.float32, resident_ctas=slots) == (units, 0, 1)


def test_backward_plan_without_a_gpu_splits_nothing(lib):
    # no device: the current-device plan splits nothing and asks for no partials
    B, H, N, d = 4, 16, 1024, 64
    assert fa.fa_bwd_plan(B, H, N, d) == (B * H * (N // 128), 0, 1)
