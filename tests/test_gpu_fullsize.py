"""Full-size parity on the benchmark workloads, in the launch configuration the
benchmark times (batched launches over all tensors of a workload).

Every tensor round-trips bit-exactly on the device; container bytes are
compared with the CPU oracle for one tensor of each shape; GEMV outputs are
checked on sampled rows that the oracle computes one by one in float64.
"""
import numpy as np
import pytest

from decode_gemv_sign_gb300 import synth
from oracle import wcomp_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMV_TOL = 1e-4


@pytest.fixture(scope="module")
def W():
    from decode_gemv_sign_gb300 import build, wcomp

    build.build()
    wcomp.lib()
    return wcomp


def host(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def sampled_gemv_check(c_ref, x_np, y_gpu, rows):
    y_ref = O.gemv_container(c_ref, x_np, rows)  # [B, len(rows)]
    y = y_gpu.cpu().numpy()[:, rows].astype(np.float64)
    scale = np.abs(y_ref).max()
    assert np.abs(y - y_ref).max() <= GEMV_TOL * scale


def run_workload(W, specs, schemes, batches, n_oracle_shapes=1, sample_rows=48):
    dev = torch.device("cuda")
    ws = [synth.gen_weights_torch(s, dev) for s in specs]
    rng = np.random.default_rng(0)
    for scheme in schemes:
        cs = [W.encode(w, scheme) for w in ws]
        outs = W.decode_batched(cs)
        for w, o in zip(ws, outs):
            assert torch.equal(w.view(-1), o.view(-1))
        del outs
        # oracle containers for the first tensor of each distinct shape
        seen = {}
        for i, s in enumerate(specs):
            if (s.N, s.K) in seen or len(seen) >= n_oracle_shapes * 2:
                continue
            w_np = host(ws[i]).reshape(s.N, s.K)
            ref = O.encode(w_np, scheme)
            assert W.serialize(cs[i]) == O.serialize(ref)
            assert W.serialize(cs[i], compact=True) == O.serialize_compact(ref)
            seen[(s.N, s.K)] = (i, ref)
        for B in batches:
            xs_np = [synth.gen_x_np(B, s.K, 9000 + i) for i, s in enumerate(specs)]
            xs = [torch.from_numpy(x.view(np.int16)).to(dev) for x in xs_np]
            ys = W.gemv_batched(cs, xs)
            for (i, ref) in seen.values():
                rows = np.sort(rng.choice(specs[i].N, size=min(sample_rows, specs[i].N), replace=False))
                sampled_gemv_check(ref, xs_np[i], ys[i], rows)
            # plain BF16 GEMV on the same inputs, same sampled rows
            for (i, ref) in seen.values():
                yp = W.gemv_bf16(ws[i], xs[i])
                rows = np.sort(rng.choice(specs[i].N, size=min(sample_rows, specs[i].N), replace=False))
                sampled_gemv_check(ref, xs_np[i], yp, rows)
        for c in cs:
            c.free()
    torch.cuda.synchronize()


def test_workload_small_full(W):
    run_workload(W, synth.workload_small(), O.SCHEMES, [1])


def test_workload_dense_layers_full(W):
    run_workload(W, synth.workload_dense_layers(), O.SCHEMES, [1, 4])


def test_workload_block6144_full(W):
    run_workload(W, synth.workload_block6144(), O.SCHEMES, [1, 4, 8, 16], sample_rows=24)


def test_workload_moe_full(W):
    """All 256 expert tensors decoded in batched launches; GEMV on the 8 chosen
    experts (both tensors each) at batch 1."""
    dev = torch.device("cuda")
    specs = synth.workload_moe()
    sel = synth.moe_selected_experts()
    for scheme in O.SCHEMES:
        ws, cs = [], []
        for s in specs:
            w = synth.gen_weights_torch(s, dev)
            cs.append(W.encode(w, scheme))
            ws.append(w)
        outs = W.decode_batched(cs)
        for w, o in zip(ws, outs):
            assert torch.equal(w.view(-1), o.view(-1))
        del outs
        idx = [2 * e + k for e in sel for k in (0, 1)]
        xs_np = [synth.gen_x_np(1, specs[i].K, 7000 + i) for i in idx]
        ys = W.gemv_batched([cs[i] for i in idx], [torch.from_numpy(x.view(np.int16)).to(dev) for x in xs_np])
        rng = np.random.default_rng(1)
        for j in (0, 1):  # one up and one down projection against the oracle
            i = idx[j]
            ref = O.encode(host(ws[i]).reshape(specs[i].N, specs[i].K), scheme)
            assert W.serialize(cs[i]) == O.serialize(ref)
            rows = np.sort(rng.choice(specs[i].N, size=32, replace=False))
            sampled_gemv_check(ref, xs_np[j], ys[j], rows)
        for c in cs:
            c.free()
        del ws
        torch.cuda.empty_cache()
