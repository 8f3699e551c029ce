"""The C ABI library without a GPU: it loads, exports every symbol the header
declares, and rejects bad arguments on the host before any CUDA call. CPU only."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

qm = pytest.importorskip("quantized_mixture_experts_route_gb300")
from quantized_mixture_experts_route_gb300 import build as qbuild  # noqa: E402


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return qm.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmoe_[a-z_]+)\s*\(", text)))


def test_exports_every_header_symbol(L):
    names = header_functions()
    assert names == sorted(qm.EXPORTED)
    for n in names:
        assert hasattr(L, n), n


def header_signatures():
    """{function: number of parameters} from the header's declarations."""
    text = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    sigs = {}
    for name, params in re.findall(r"\b(qmoe_[a-z_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = params.strip()
        sigs[name] = 0 if params in ("", "void") else params.count(",") + 1
    return sigs


def test_binding_argument_counts_match_header(L):
    sigs = header_signatures()
    assert sorted(sigs) == sorted(qm.EXPORTED)
    for name, n in sigs.items():
        assert len(getattr(L, name).argtypes) == n, name


def test_status_strings(L):
    for s in range(6):
        assert qm.qmoe_status_string(s)
    assert "unknown" in qm.qmoe_status_string(99)


def P(**kw):
    base = dict(T=8, hidden=2048, inter=768, num_experts=128, top_k=8, bits=4, block_size=32,
                dtype=qm.QMOE_BF16, path=qm.QMOE_PATH_AUTO)
    base.update(kw)
    return qm.problem(**base)


BAD = [
    (dict(num_experts=0), qm.QMOE_ERR_INVALID_ARGUMENT),
    (dict(top_k=0), qm.QMOE_ERR_INVALID_ARGUMENT),
    (dict(top_k=129), qm.QMOE_ERR_INVALID_ARGUMENT),
    (dict(hidden=0), qm.QMOE_ERR_INVALID_ARGUMENT),
    (dict(inter=-32), qm.QMOE_ERR_INVALID_ARGUMENT),
    (dict(T=-1), qm.QMOE_ERR_INVALID_ARGUMENT),
    (dict(bits=5), qm.QMOE_ERR_UNSUPPORTED),
    (dict(bits=8), qm.QMOE_ERR_UNSUPPORTED),
    (dict(block_size=16), qm.QMOE_ERR_UNSUPPORTED),
    (dict(block_size=128, inter=704), qm.QMOE_ERR_UNSUPPORTED),
    (dict(hidden=2056), qm.QMOE_ERR_UNSUPPORTED),
    (dict(num_experts=1024, top_k=8), qm.QMOE_ERR_UNSUPPORTED),
    (dict(num_experts=64, top_k=33), qm.QMOE_ERR_UNSUPPORTED),
    (dict(dtype=2), qm.QMOE_ERR_UNSUPPORTED),
    (dict(path=5), qm.QMOE_ERR_UNSUPPORTED),
    (dict(path=qm.QMOE_PATH_GROUPED_WS, T=64, hidden=96, inter=64), qm.QMOE_ERR_UNSUPPORTED),
    (dict(path=qm.QMOE_PATH_GROUPED_WS, T=64, hidden=320, inter=256), qm.QMOE_ERR_UNSUPPORTED),   # 256 | H
    (dict(path=qm.QMOE_PATH_DECODE, T=65), qm.QMOE_ERR_UNSUPPORTED),
    (dict(path=qm.QMOE_PATH_DECODE, T=64, top_k=16), qm.QMOE_ERR_UNSUPPORTED),   # 1024 routes
    (dict(path=qm.QMOE_PATH_GROUPED, bits=3, block_size=64, hidden=2048, inter=704), qm.QMOE_ERR_UNSUPPORTED),
    (dict(T=64, hidden=96, inter=64), qm.QMOE_ERR_UNSUPPORTED),   # grouped path: multiples of 64
]

FAKE = 1 << 20  # an aligned address that is never dereferenced: every call below fails its checks first


def call_forward(L, p, ptrs=None, ws_bytes=1 << 40, misalign=None, ex=False):
    args = [FAKE] * 10 if ptrs is None else list(ptrs)
    if misalign is not None:
        args[misalign] += 2
    if ex:   # qmoe_forward_ex with default options makes the same checks
        opt = qm.qmoe_options(0, None, None)
        return L.qmoe_forward_ex(ctypes.byref(p), ctypes.byref(opt), *args[:9], args[9], ws_bytes, None)
    return L.qmoe_forward(ctypes.byref(p), *args[:9], args[9], ws_bytes, None)


@pytest.mark.parametrize("kw,status", BAD, ids=[str(b[0]) for b in BAD])
def test_invalid_problem_rejected(L, kw, status):
    p = P(**kw)
    assert call_forward(L, p) == status
    assert call_forward(L, p, ex=True) == status
    assert L.qmoe_route(ctypes.byref(p), FAKE, None, None, None, None, FAKE, 1 << 40, None) == status
    assert L.qmoe_workspace_bytes(ctypes.byref(p)) == 0


def test_null_problem(L):
    assert L.qmoe_forward(None, *([FAKE] * 10), 1 << 40, None) == qm.QMOE_ERR_INVALID_ARGUMENT
    assert L.qmoe_workspace_bytes(None) == 0


@pytest.mark.parametrize("which", [0, 1, 2, 3, 5, 6, 8, 9])
def test_null_required_pointer(L, which):
    args = [FAKE] * 10
    args[which] = None
    assert call_forward(L, P(), args) == qm.QMOE_ERR_INVALID_ARGUMENT
    assert call_forward(L, P(), args, ex=True) == qm.QMOE_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("which", range(10))
def test_misaligned_pointer(L, which):
    assert call_forward(L, P(), misalign=which) == qm.QMOE_ERR_MISALIGNED
    assert call_forward(L, P(), misalign=which, ex=True) == qm.QMOE_ERR_MISALIGNED


def test_workspace_too_small(L):
    p = P()
    need = L.qmoe_workspace_bytes(ctypes.byref(p))
    assert need > 0
    assert call_forward(L, p, ws_bytes=need - 1) == qm.QMOE_ERR_WORKSPACE_TOO_SMALL
    assert call_forward(L, p, ws_bytes=need - 1, ex=True) == qm.QMOE_ERR_WORKSPACE_TOO_SMALL
    assert L.qmoe_route(ctypes.byref(p), FAKE, None, None, None, None, FAKE, need - 1, None) == \
        qm.QMOE_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("field,value", [("full_softmax", 2), ("full_softmax", -1),
                                         ("decode_layer_kernel", 2), ("decode_layer_kernel", -1)])
def test_invalid_option_rejected(L, field, value):
    """Option values other than 0 and 1 are refused before anything is read or launched."""
    opt = qm.qmoe_options(0, None, None, 0)
    setattr(opt, field, value)
    args = [FAKE] * 10
    assert L.qmoe_forward_ex(ctypes.byref(P()), ctypes.byref(opt), *args[:9], args[9], 1 << 40, None) == \
        qm.QMOE_ERR_INVALID_ARGUMENT


def test_options_struct_matches_the_header():
    """The binding's qmoe_options has the header's fields, in order."""
    import os
    import re

    from tests.conftest import ROOT

    hdr = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    body = re.search(r"typedef struct \{([^}]*)\} qmoe_options;", hdr).group(1)
    names = re.findall(r"(\w+);", body)
    assert names == [f[0] for f in qm.qmoe_options._fields_]


@pytest.mark.parametrize("kw,path", [
    (dict(T=8), "decode"),
    (dict(T=16), "decode"),                            # 128 routes < 4 E = 512
    (dict(T=63), "decode"),                            # 504 routes
    (dict(T=64), "grouped"),                           # 512 routes = 4 E: the pages' switch
    (dict(T=9, num_experts=4, top_k=2), "decode"),     # 18 routes < 64
    (dict(T=40, num_experts=8, top_k=2), "grouped"),   # 80 routes >= 64 and >= 4 E
    (dict(T=64, num_experts=512, top_k=8), "decode"),  # 512 routes < 4 E
    (dict(T=48, num_experts=512, top_k=16), "grouped"),  # 768 routes: above one grouping block
])
def test_auto_path_follows_the_route_count(L, kw, path):
    """AUTO takes the decode path for T <= 8 and, up to 64 tokens and 512 routes, while
    the routes number fewer than 64 or fewer than 4 per expert; the path shows in the
    workspace size (the grouped path adds the gathered activation rows)."""
    auto = L.qmoe_workspace_bytes(ctypes.byref(P(**kw)))
    want = L.qmoe_workspace_bytes(ctypes.byref(P(**kw, path=qm.QMOE_PATH_DECODE if path == "decode"
                                                       else qm.QMOE_PATH_GROUPED)))
    other = L.qmoe_workspace_bytes(ctypes.byref(P(**kw, path=qm.QMOE_PATH_GROUPED if path == "decode"
                                                        else qm.QMOE_PATH_DECODE)))
    assert auto == want > 0 and auto != other


def test_empty_input_is_noop(L):
    # T == 0: OK with no launch, even with null buffers
    p = P(T=0)
    assert L.qmoe_forward(ctypes.byref(p), *([None] * 10), 0, None) == qm.QMOE_OK
    assert L.qmoe_route(ctypes.byref(p), None, None, None, None, None, None, 0, None) == qm.QMOE_OK


def test_workspace_sizes_grow_with_T(L):
    small = L.qmoe_workspace_bytes(ctypes.byref(P(T=1)))
    dec = L.qmoe_workspace_bytes(ctypes.byref(P(T=8)))
    pre = L.qmoe_workspace_bytes(ctypes.byref(P(T=8192)))
    assert 0 < small < dec < pre
    # the grouped layout at 8K: x16 + gathered x16 + h16 + FP32 y dominate
    R = 8192 * 8
    assert pre >= R * (2048 * 2 + 768 * 2 + 2048 * 4)


@pytest.mark.parametrize("first,last", [(-1, 3), (0, 4), (2, 1)])
def test_bad_stage_range(L, first, last):
    p = P()
    assert L.qmoe_forward_stages(ctypes.byref(p), first, last, *([FAKE] * 10), 1 << 40, None) == \
        qm.QMOE_ERR_INVALID_ARGUMENT


def test_launch_facts_are_per_device():
    """The shared-memory opt-in and the SM count belong to a device's context:
    the launchers look them up through one per-(device, context) cache, and no
    launcher keeps a process-wide flag or count of its own."""
    csrc = os.path.join(ROOT, "quantized_mixture_experts_route_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh")) or name == "launch_cache.cu":
            continue
        code = "\n".join(line.split("//")[0] for line in open(os.path.join(csrc, name)).read().splitlines())
        assert not re.search(r"\bstatic\s+(bool|int)\s+\w+\s*=", code), f"{name}: process-wide launch state"
        assert "cudaFuncSetAttribute" not in code, f"{name}: opt-in outside the per-device cache"
        assert "cudaDevAttrMultiProcessorCount" not in code, f"{name}: SM count outside the per-device cache"
