"""The bench's count of our kernels per step (its `gpu_launches` claim), checked
on the CPU against the kernels ncu listed for each named workload on a 152-SM
GB300: kv_write, the plan kernel (not when the decode kernel plans the call
itself), decode, the tensor-core chunk kernel (a request with more than 64
rows), the shared-prefix pass (a shared table prefix), combine."""

import pytest

import bench
import workloads as wl

# kernels per step, bf16 and E4M3 caches alike, from the launch lists
EXPECTED = {
    "tiny-decode": 3,         # kv_write, decode (plans itself), combine
    "tinyllama-decode": 3,    # kv_write, decode (plans itself), combine
    "llama13b-decode": 4,     # kv_write, plan, decode, combine
    "llama3-8b-mixed": 5,     # kv_write, plan, decode, chunk kernel, combine
    "llama3-70b-prefix": 5,   # kv_write, plan, decode, shared-prefix pass, combine
}


@pytest.mark.parametrize("name", sorted(EXPECTED))
@pytest.mark.parametrize("fp8", [False, True])
def test_kernels_per_step_match_the_launch_lists(name, fp8):
    step = wl.make_workload(name)
    K = bench.shared_prefix_blocks(step)
    assert bench.launches_per_step(step, K, fp8, 152) == EXPECTED[name]


def test_self_planned_decode_follows_the_batch_bound():
    # the same batch shape with more requests than the decode grid's warps can
    # take as (request, kv head) pairs goes through the plan kernel
    small = wl.make_workload("tinyllama-decode")
    assert bench.decode_self_planned(small, 0, False, 152)
    assert not bench.decode_self_planned(small, 8, False, 152)      # a shared prefix: the plan kernel
    assert not bench.decode_self_planned(wl.make_workload("llama13b-decode"), 0, False, 152)


def test_traffic_keys_name_the_kernels_of_the_call():
    assert bench.traffic_key(wl.make_workload("llama13b-decode"), False, 0) == "bf16 decode"
    assert bench.traffic_key(wl.make_workload("llama3-8b-mixed"), True, 0) == "e4m3 prefill"
    prefix = wl.make_workload("llama3-70b-prefix")
    assert bench.traffic_key(prefix, False, bench.shared_prefix_blocks(prefix)) == "bf16 cascade"
