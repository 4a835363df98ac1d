import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def _device_line():
    try:
        import torch
        if torch.cuda.is_available():
            p = torch.cuda.get_device_properties(0)
            return f"cuda device 0: {p.name}, {p.multi_processor_count} SMs, torch {torch.__version__}"
    except Exception as e:  # a report line only; never fails the run
        return f"cuda device 0: unknown ({e})"
    return None


def pytest_report_header(config):
    return _device_line()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    line = _device_line()
    if line:
        terminalreporter.write_line(line)
