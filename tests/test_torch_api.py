"""The tensor-level calls (collective_datapath_atom_gb300.torch_api): argument
checks on the CPU, and on a GPU every collective against the CPU oracle."""
import numpy as np
import pytest

import oracle
from test_parity_gpu import gen_inputs

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def T():
    import __graft_entry__

    __graft_entry__.build()
    from collective_datapath_atom_gb300 import torch_api

    return torch_api


class FakeHandle:
    R = 4


def test_dtype_inference(T):
    f32 = [torch.zeros(4, dtype=torch.float32) for _ in range(2)]
    bf = [torch.zeros(4, dtype=torch.bfloat16) for _ in range(2)]
    bits = [torch.zeros(4, dtype=torch.int16) for _ in range(2)]
    assert T._dtype_of(f32) == 0 and T._dtype_of(bf) == 1 and T._dtype_of(bits) == 1
    with pytest.raises(TypeError):
        T._dtype_of([torch.zeros(4, dtype=torch.float16)])
    with pytest.raises(TypeError):
        T._dtype_of(f32[:1] + bf[:1])


def test_argument_checks_without_a_gpu(T):
    xs = [torch.zeros(8) for _ in range(4)]
    with pytest.raises(ValueError):           # wrong number of ranks
        T._check(xs[:3], xs, FakeHandle())
    with pytest.raises(ValueError):           # host tensors
        T._check(xs, xs, FakeHandle())
    with pytest.raises(ValueError):
        T._uniform_numel([torch.zeros(3), torch.zeros(4)])
    with pytest.raises(NotImplementedError):  # no NVLS on one GPU
        T.all_reduce(xs, xs, FakeHandle(), reduction_mode=T.ReductionMode.NON_DETERMINISTIC)


@pytest.mark.gpu
def test_every_collective_through_the_tensor_calls(T):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    R = 4
    stream = torch.cuda.current_stream()
    h = T.initialize(R, stream=stream)
    try:
        def dev(arrs):
            return [torch.from_numpy(a.view(np.int16).copy()).cuda() for a in arrs]

        def host(ts):
            return [t.cpu().numpy().view(np.uint16) for t in ts]

        n = 4096 + 8
        ins = gen_inputs([n] * R, 1, seed=1)
        xs = dev(ins)
        outs = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)]
        T.all_reduce(xs, outs, h, stream=stream)
        assert all(np.array_equal(g, w) for g, w in zip(host(outs), oracle.all_reduce(ins, 1)))
        outs = [torch.empty(n // R, dtype=torch.int16, device="cuda") for _ in range(R)]
        T.reduce_scatter(xs, outs, h)
        assert all(np.array_equal(g, w) for g, w in zip(host(outs), oracle.reduce_scatter(ins, 1)))
        outs = [torch.empty(R * n, dtype=torch.int16, device="cuda") for _ in range(R)]
        T.all_gather(xs, outs, h)
        assert all(np.array_equal(g, w) for g, w in zip(host(outs), oracle.all_gather(ins, 1)))
        outs = [torch.empty(n, dtype=torch.int16, device="cuda") for _ in range(R)]
        T.all_to_all(xs, outs, h)
        assert all(np.array_equal(g, w) for g, w in zip(host(outs), oracle.all_to_all(ins, 1)))
        counts = [100, 7, 0, 2049]
        vins = gen_inputs(counts, 1, seed=2)
        outs = [torch.empty(sum(counts), dtype=torch.int16, device="cuda") for _ in range(R)]
        T.all_gather_v(dev(vins), outs, h)
        assert all(np.array_equal(g, w)
                   for g, w in zip(host(outs), oracle.all_gather_v(vins, counts, 1)))
        rins = gen_inputs([sum(counts)] * R, 1, seed=3)
        outs = [torch.empty(c, dtype=torch.int16, device="cuda") for c in counts]
        T.reduce_scatter_v(dev(rins), outs, h)
        assert all(np.array_equal(g, w)
                   for g, w in zip(host(outs), oracle.reduce_scatter_v(rins, counts, 1)))
        C = np.array([[3, 0, 5, 1], [2, 2, 2, 2], [0, 0, 0, 9], [7, 1, 0, 0]])
        ains = gen_inputs([int(C[s].sum()) for s in range(R)], 1, seed=4)
        outs = [torch.empty(int(C[:, d].sum()), dtype=torch.int16, device="cuda")
                for d in range(R)]
        T.all_to_all_v(dev(ains), outs, C.tolist(), h)
        assert all(np.array_equal(g, w)
                   for g, w in zip(host(outs), oracle.all_to_all_v(ains, C, 1)))
        T.check(h)
    finally:
        T.finalize(h)
